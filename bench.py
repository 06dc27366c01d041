#!/usr/bin/env python
"""Benchmark of the verify hot path on GB300.

Workload (one step): the dense-27B-like layer verify -- d = 5120; q, k, v, o
(5120 -> 6144 / 1024 / 1024, 6144 -> 5120), gate and up (5120 -> 17408) and
down (17408 -> 5120) -- as nvfp4 weights (N(0, 0.02) quantized), with M = 8
bf16 N(0, 1) verify rows.  q/k/v and gate/up read the same input and are
stored concatenated along N, as inference engines store them, so the step is
four verify_gemm_w4 calls back to back on one stream (qkv 5120 -> 8192, o,
gate_up 5120 -> 34816, down).  The weights and scales of one step (191.7 MB)
exceed the 129 MB L2, so every step streams them from HBM.

Metric: HBM GB/s = algorithmic bytes (packed weights + scales + activations)
per step / step time, summed over ranks (N independent replicas).  The same
JSON line carries the per-M microseconds for M = 1, 2, 4, 8 (nvfp4 and Q4_0),
the seven-call (unpacked) layer for comparison, the accept-step
microseconds, the roofline of the GEMM kernel, the end-to-end number through
the C ABI with host buffers, the CPU oracle baseline and the SM clocks seen
during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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

import numpy as np  # noqa: E402

# The seven linears of the layer, and the step as an inference engine stores
# them: q/k/v and gate/up each read the same input, so their weights sit
# concatenated along N (one packed matrix, one call each).  The packed step
# streams the same weight bytes with 4 calls instead of 7.
LAYER = [("q", 6144, 5120), ("k", 1024, 5120), ("v", 1024, 5120), ("o", 5120, 6144),
         ("gate", 17408, 5120), ("up", 17408, 5120), ("down", 5120, 17408)]
STEP = [("qkv", 8192, 5120), ("o", 5120, 6144), ("gate_up", 34816, 5120), ("down", 5120, 17408)]
HEAD_M = 8
# verify widths timed per M (9..16 rows take the two-n-tile kernel)
PER_M = (1, 2, 4, 8, 16)
METRIC = "nvfp4 verify-GEMM HBM GB/s & µs/pass at M=1,2,4,8; accept µs/step"
WORKLOAD = ("dense-27B-like layer verify: d=5120, q/k/v/o 5120->6144/1024/1024 and 6144->5120, "
            "gate/up 5120->17408, down 17408->5120, nvfp4 (E2M1 + E4M3 per 16 + fp32 tensor "
            "scale), bf16 activations N(0,1), M=8 verify rows; q/k/v and gate/up packed along "
            "N (qkv 5120->8192, gate_up 5120->34816): 4 verify_gemm_w4 calls per step")
SPEC_HBM_GBS = 8000.0
LAUNCHES_PER_GEMM = 2   # activation prep + the GEMM kernel


def weight_bytes(N, K, fmt="nvfp4"):
    return N * K // 2 + (N * K // 16 if fmt == "nvfp4" else N * K // 32 * 2)


def step_bytes(M, fmt="nvfp4", spec=None):
    return sum(weight_bytes(N, K, fmt) + M * K * 2 for _, N, K in (spec or STEP))


KERNEL_SOURCES = ["speculative_decode_verification_w4_gb300/csrc/" + f
                  for f in ("gemm_w4.cu", "vw4_internal.cuh", "ptx.cuh", "api.cu")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_w4_dense_layer_m8_traffic.json")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic():
    """DRAM bytes (read + write) of the GEMM kernel per layer step (its 4
    launches), from the committed ncu summary -- null when the kernel sources
    changed since those counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_step")


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed loop runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                    "raw": self.lines[:2]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ inputs
def make_layer(fmt, device, spec=None):
    import torch
    import synth
    layer = []
    for i, (name, N, K) in enumerate(spec or STEP):
        q, s, ts = synth.linear(100 + i, N, K, fmt)
        qd = torch.from_numpy(q).to(device)
        if fmt == "nvfp4":
            sd = torch.from_numpy(s).to(device)
        else:
            sd = torch.from_numpy(s.view(np.uint16)).to(device).view(torch.float16)
        layer.append((name, N, K, qd, sd, ts))
    return layer


def make_acts(M, device, seed=7, spec=None):
    import torch
    import synth
    g = synth.rng(seed)
    acts = []
    for _, N, K in (spec or STEP):
        bits = synth.activations(g, M, K)
        acts.append(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device))
    return acts


# --------------------------------------------------------------- our arm
def run_ours(args, rank, world, device):
    import torch
    import speculative_decode_verification_w4_gb300 as vw4

    torch.cuda.set_device(device)
    layers = {"nvfp4": make_layer("nvfp4", device), "q4_0": make_layer("q4_0", device)}
    # a second copy of the nvfp4 layer: the headline alternates the two, so
    # that 383 MB of weights (more than twice the 129 MB L2) pass per two steps
    layer_b = [(name, N, K, qd.clone(), sd.clone(), ts) for (name, N, K, qd, sd, ts) in
               layers["nvfp4"]]
    acts = {M: make_acts(M, device, seed=7 + M) for M in PER_M}
    outs = {M: [torch.empty((M, N), dtype=torch.float32, device=device) for _, N, _ in STEP]
            for M in PER_M}
    ws = vw4.Workspace(device)
    ws.get(max(vw4.vw4_workspace_bytes(vw4.OP_GEMM, max(PER_M), N, K)
               for _, N, K in STEP + LAYER))
    FMTS = {"nvfp4": vw4.FMT_NVFP4, "q4_0": vw4.FMT_Q4_0}

    def one_step(fmt, M, layer=None):
        for j, (name, N, K, qd, sd, ts) in enumerate(layer or layers[fmt]):
            vw4.verify_gemm_w4(FMTS[fmt], qd, sd, ts, acts[M][j], out=outs[M][j], workspace=ws)

    def capture(fn, warm=3):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def time_graph(g, reps, warmup, g_alt=None):
        """ms for reps replays (alternating g and g_alt when given)."""
        seq = [g, g_alt] if g_alt is not None else [g]
        for i in range(warmup):
            seq[i % len(seq)].replay()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(reps):
            seq[i % len(seq)].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return e0.elapsed_time(e1)

    def time_steps(g_pair, g_one, n, warmup):
        """ms for exactly n steps: n // 2 replays of the two-step graph, then
        the one-step graph if n is odd (after ceil(warmup / 2) pair replays)."""
        for _ in range((warmup + 1) // 2):
            g_pair.replay()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n // 2):
            g_pair.replay()
        if n % 2:
            g_one.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return e0.elapsed_time(e1)

    def time_alone(fmt, name, N, K, qd, sd, ts, A, out, steps):
        """One call timed alone: a graph of R calls on R different weight copies
        (more than 2x L2 of weights in flight, so nothing is served from L2)."""
        R = max(4, int(np.ceil(320e6 / weight_bytes(N, K, fmt))))
        copies = [(qd.clone(), sd.clone()) for _ in range(R)]

        def calls():
            for (qc, sc) in copies:
                vw4.verify_gemm_w4(FMTS[fmt], qc, sc, ts, A, out=out, workspace=ws)
        gl = capture(calls, warm=1)
        reps = max(2, int(np.ceil(steps / 4)))
        us = time_graph(gl, reps, 1) / (reps * R) * 1e3
        del gl, copies
        torch.cuda.empty_cache()
        return round(us, 2)

    steps, warmup = args.steps, args.warmup
    peak, peak_kind = read_peaks()
    with ClockSampler(torch.cuda.current_device()) as clk:
        # headline: one step = the packed layer at M = 8 (the four C-ABI
        # calls).  Consecutive steps alternate the two weight copies and are
        # captured in pairs, one CUDA graph per pair, as an engine captures
        # consecutive layers in one graph; an odd K ends on a one-step graph.
        def two_steps():
            one_step("nvfp4", HEAD_M)
            one_step("nvfp4", HEAD_M, layer_b)
        g_head = capture(lambda: one_step("nvfp4", HEAD_M))
        g_pair = capture(two_steps)
        soak_end = time.time() + 0.4
        while time.time() < soak_end:      # let the clock sampler see the load
            for _ in range(10):
                g_pair.replay()
            torch.cuda.synchronize()
        ms = time_steps(g_pair, g_head, steps, warmup)
        ms_max = reduce_max(ms, world)
        ms_per_step = ms_max / steps
        value = step_bytes(HEAD_M) * steps * world / (ms_max * 1e-3) / 1e9

        # per-M microseconds of the packed layer (graph of the step), both
        # formats, and of each of its calls alone
        per_m = {}
        for fmt in ("nvfp4", "q4_0"):
            per_m[fmt] = {}
            for M in PER_M:
                gm = capture(lambda: one_step(fmt, M))
                m_ms = time_graph(gm, steps, 3)
                per_m[fmt][str(M)] = {
                    "layer_us": round(m_ms / steps * 1e3, 2),
                    "layer_gbs": round(step_bytes(M, fmt) / (m_ms / steps * 1e-3) / 1e9, 1),
                    "call_us": {}}
                del gm
            for j, (name, N, K, qd, sd, ts) in enumerate(layers[fmt]):
                for M in PER_M:
                    per_m[fmt][str(M)]["call_us"][name] = time_alone(
                        fmt, name, N, K, qd, sd, ts, acts[M][j], outs[M][j], steps)

        # the same layer as seven separate calls (no packing), nvfp4
        unpacked = {}
        lay7 = make_layer("nvfp4", device, LAYER)
        for M in (1, 8):
            a7 = make_acts(M, device, seed=17 + M, spec=LAYER)
            o7 = [torch.empty((M, N), dtype=torch.float32, device=device) for _, N, _ in LAYER]

            def step7(a7=a7, o7=o7):
                for j, (name, N, K, qd, sd, ts) in enumerate(lay7):
                    vw4.verify_gemm_w4(vw4.FMT_NVFP4, qd, sd, ts, a7[j], out=o7[j], workspace=ws)
            g7 = capture(step7)
            m7 = time_graph(g7, steps, 3)
            del g7
            unpacked[str(M)] = {
                "layer_us": round(m7 / steps * 1e3, 2),
                "layer_gbs": round(step_bytes(M, "nvfp4", LAYER) / (m7 / steps * 1e-3) / 1e9, 1),
                "linear_us": {name: time_alone("nvfp4", name, N, K, qd, sd, ts, a7[j], o7[j], steps)
                              for j, (name, N, K, qd, sd, ts) in enumerate(lay7)}}
        del lay7
        torch.cuda.empty_cache()

    stream = torch.cuda.current_stream()
    accept = run_accept_timings(device, stream)
    heads = run_head_timings(device, stream)
    gate = {}
    for name in ("qkv", "o", "gate_up", "down"):
        t1 = per_m["nvfp4"]["1"]["call_us"][name]
        t8 = per_m["nvfp4"]["8"]["call_us"][name]
        N, K = [(n, k) for nm, n, k in STEP if nm == name][0]
        gbs = (weight_bytes(N, K) + 8 * K * 2) / (t8 * 1e-6) / 1e9
        gate[name] = {"m8_over_m1": round(t8 / t1, 3), "m8_gbs": round(gbs, 1),
                      "frac_of_8tbs": round(gbs / SPEC_HBM_GBS, 3),
                      "frac_of_measured_copy": round(gbs / peak, 3)}

    lm = heads.get("lmhead_per_m") if isinstance(heads, dict) else None
    if lm:
        t1, t8 = lm["1"]["us"], lm["8"]["us"]
        gbs = lm["8"]["gbs"]
        gate["lm_head"] = {"m8_over_m1": round(t8 / t1, 3), "m8_gbs": gbs,
                           "frac_of_8tbs": round(gbs / SPEC_HBM_GBS, 3),
                           "frac_of_measured_copy": round(gbs / peak, 3)}

    # roofline of the GEMM: algorithmic bytes of the step's calls at M = 8 over
    # their times, each call timed alone (graph replay, CUDA events)
    t_call = per_m["nvfp4"]["8"]["call_us"]
    achieved = step_bytes(HEAD_M) / (sum(t_call[n] for n, _, _ in STEP) * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": measured_traffic(),
                "per": "layer step: the 4 GEMM calls at M = 8 (bytes, time, traffic)",
                "peak_kind": f"of {peak_kind} (STREAM-style copy, burst)",
                "kernel": "vw4::gemm_w4_kernel<nvfp4> (with its activation-prep launch)",
                "per_unit": "0.5625 B per weight (nibble + e4m3/16) + 2*M B per k of activations"}

    depth = depth_controller_summary(per_m)

    e2e = run_e2e(vw4, layers["nvfp4"], layer_b, device, steps, warmup, world)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 x f16 -> f32 (exact nibble*scale products, fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": HEAD_M, "fmt": "nvfp4",
                   "bytes_per_step": step_bytes(HEAD_M),
                   "l2": "inputs larger than L2: 191.7 MB of weights+scales per step, two "
                         "weight copies alternating (383 MB per two steps) vs 129 MB L2",
                   "timing": "one CUDA graph per two consecutive steps (the 4 C-ABI calls on "
                             "weight copy A, then on copy B), replayed back to back; an odd "
                             "step count ends on a one-step graph",
                   "parallelism": f"replicas x{world}"},
        "per_m": per_m, "unpacked_7_calls": unpacked, "gate": gate, "accept_us": accept,
        "depth_controller": depth,
        "heads": heads,
        "roofline": roofline, "e2e": e2e,
        "gpu_launches": steps * len(STEP) * LAUNCHES_PER_GEMM,
        "clocks": clk.summary(),
    }
    return result


def depth_controller_summary(per_m):
    """The draft-depth controller on the measured verify cost of each width
    (the nvfp4 layer step at the measured M, linear in between), a synthetic
    acceptance of 0.8 at every position and, as an assumption, a draft
    costing a tenth of a one-row verify step per token."""
    import speculative_decode_verification_w4_gb300 as vw4
    mus = {int(m): per_m["nvfp4"][m]["layer_us"] for m in per_m["nvfp4"]}
    pts = sorted(mus)
    k_max = max(pts) - 1
    verify_us = {w: float(np.interp(w, pts, [mus[p] for p in pts])) for w in range(1, k_max + 2)}
    ctl = vw4.DepthController(k_max=k_max, decay=1.0, verify_us=verify_us,
                              draft_us_per_token=0.1 * verify_us[1])
    for i in range(k_max + 1):  # counts giving (acc + 1) / (att + 2) ~ 0.8 at every position
        ctl.state.att[i], ctl.state.acc[i] = 10000.0, 8000.0
    rates = {k: round(ctl.expected(k)[0] / ctl.expected(k)[1] * 1e3, 3)
             for k in range(k_max + 1)}
    return {"acceptance": 0.8, "draft_us_per_token": round(0.1 * verify_us[1], 2),
            "verify_us": {w: round(v, 2) for w, v in verify_us.items()},
            "committed_tokens_per_ms": rates, "chosen_depth": ctl.choose()}


def run_accept_timings(device, stream):
    """accept_rejection on the stochastic sweep (B=256, V=151936, K=1,4,8) and
    accept_greedy on LM-head-sized logits (B=1, 7 drafts, V=262144)."""
    import torch
    import speculative_decode_verification_w4_gb300 as vw4
    out = {}
    g = torch.Generator(device=device).manual_seed(4)
    B, V = 256, 151936
    for Kd in (1, 4, 8):
        tgt = torch.randn((B, Kd + 1, V), generator=g, device=device) * 3.0
        drf = tgt[:, :Kd] + torch.randn((B, Kd, V), generator=g, device=device)
        probs = torch.softmax(drf.reshape(-1, V) / 0.6, dim=-1)
        drafts = torch.multinomial(probs, 1, generator=g).reshape(B, Kd).to(torch.int32)
        del probs
        ws = vw4.Workspace(device)
        for _ in range(3):
            vw4.accept_rejection(tgt, drf, drafts, 0.6, 0.95, 4, 0, workspace=ws, stream=stream)
        torch.cuda.synchronize()
        reps = 10
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for r in range(reps):
            vw4.accept_rejection(tgt, drf, drafts, 0.6, 0.95, 4, r, workspace=ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        out[f"rejection_K{Kd}"] = {"us": round(us, 1),
                                   "logit_gbs": round(B * (2 * Kd + 1) * V * 4 / (us * 1e-6) / 1e9, 1)}
        if Kd in (1, 8):
            # the same step with the sampler's top-k (50) and min-p (0.05) stages on
            e0.record(stream)
            for r in range(reps):
                vw4.accept_rejection(tgt, drf, drafts, 0.6, 0.95, 4, r, top_k=50, min_p=0.05,
                                     workspace=ws, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) / reps * 1e3
            out[f"rejection_K{Kd}_topk50_minp0.05"] = {
                "us": round(us, 1),
                "logit_gbs": round(B * (2 * Kd + 1) * V * 4 / (us * 1e-6) / 1e9, 1)}
            # the rows handed on as top-64 lists (ids and logits; taken here
            # with torch.topk, outside the timed region) to accept_rejection_topk,
            # with drafts drawn from the draft lists; the lists (2.2 MB at K = 8)
            # stay in L2 across the repetitions
            Kt = 64
            tv, ti = torch.topk(tgt, Kt, dim=-1)
            dv, di = torch.topk(drf, Kt, dim=-1)
            ti, di = ti.to(torch.int32).contiguous(), di.to(torch.int32).contiguous()
            tv, dv = tv.contiguous(), dv.contiguous()
            pick = torch.multinomial(torch.softmax(dv.reshape(-1, Kt) / 0.6, dim=-1), 1,
                                     generator=g).reshape(B, Kd, 1)
            ldrafts = torch.gather(di, 2, pick).reshape(B, Kd).contiguous()
            for _ in range(3):
                vw4.accept_rejection_topk(ti, tv, di, dv, ldrafts, V, 0.6, 0.95, 4, 0,
                                          workspace=ws, stream=stream)
            torch.cuda.synchronize()
            e0.record(stream)
            for r in range(reps):
                vw4.accept_rejection_topk(ti, tv, di, dv, ldrafts, V, 0.6, 0.95, 4, r,
                                          workspace=ws, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) / reps * 1e3
            out[f"rejection_topk_lists_K{Kd}_kt{Kt}"] = {
                "us": round(us, 1), "list_bytes": B * (2 * Kd + 1) * Kt * 8}
            del tv, ti, dv, di
        del tgt, drf
    # greedy accept of 7 drafts from 8 fp32 logits rows of the LM head (V =
    # 262144): a CUDA graph over 20 logits copies (160 MB, more than L2), so
    # that neither host launch work nor L2 residency enters the number
    V, n_copy = 262144, 20
    lgs = [torch.randn((1, 8, V), generator=g, device=device) for _ in range(n_copy)]
    drafts = torch.argmax(lgs[0][:, :7], dim=-1).to(torch.int32)
    tk = torch.empty((1, 8), dtype=torch.int32, device=device)
    ln = torch.empty((1,), dtype=torch.int32, device=device)
    gs = torch.cuda.Stream(device)
    for lg in lgs:
        vw4.accept_greedy(lg, drafts, tokens=tk, length=ln, stream=gs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for lg in lgs:
            vw4.accept_greedy(lg, drafts, tokens=tk, length=ln, stream=gs)
    reps = 10
    with torch.cuda.stream(gs):
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(gs)
        for _ in range(reps):
            graph.replay()
        e1.record(gs)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / (reps * n_copy) * 1e3
    out["greedy_lmhead_unfused"] = {"us": round(us, 2),
                                    "logit_gbs": round(8 * V * 4 / (us * 1e-6) / 1e9, 1)}
    del lgs
    torch.cuda.empty_cache()
    return out


def run_head_timings(device, stream):
    """The two other verify configurations, timed with CUDA events:
    * MoE head: 128 experts, top-8, d = 2048, expert gate/up 2048 -> 768 each
      (stacked) and down 768 -> 2048, nvfp4, M = 8 tokens with seeded top-8
      routing: the pair GEMM and the down GEMM with the gate combine (the
      silu(gate) * up between them is harness work, made once);
    * LM head 5376 -> 262144 nvfp4, M = 8, with the fused argmax, and the
      greedy accept of 7 drafts from that argmax.
    Two weight copies alternate, so that nothing is served from L2."""
    import torch
    import synth
    import speculative_decode_verification_w4_gb300 as vw4
    out = {}
    stream = torch.cuda.Stream(device)  # graphs are captured off the default stream
    torch.cuda.synchronize()
    E, d, f, M, topk = 128, 2048, 768, 8, 8
    gu = [synth.linear(200 + c, E * 2 * f, d, "nvfp4") for c in range(2)]
    dn = [synth.linear(210 + c, E * d, f, "nvfp4") for c in range(2)]
    gu = [(torch.from_numpy(q).to(device), torch.from_numpy(sc).to(device), ts) for q, sc, ts in gu]
    dn = [(torch.from_numpy(q).to(device), torch.from_numpy(sc).to(device), ts) for q, sc, ts in dn]
    ids, gates = synth.routing(300, M, E, topk)
    ids_d = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).to(device)
    gates_d = torch.from_numpy(np.ascontiguousarray(gates, np.float32)).to(device)
    A = torch.from_numpy(synth.activations(synth.rng(301), M, d).view(np.int16)).view(
        torch.bfloat16).to(device)
    pair = torch.empty((M * topk, 2 * f), dtype=torch.float32, device=device)
    res = torch.empty((M, d), dtype=torch.float32, device=device)
    g0, u0 = pair[:, :f], pair[:, f:]
    ws = vw4.Workspace(device)
    vw4.verify_moe_w4(vw4.FMT_NVFP4, *gu[0], E, A, 0, ids_d, gates_d, 0, out=pair, workspace=ws,
                      stream=stream)
    h = (torch.nn.functional.silu(g0) * u0).to(torch.bfloat16).contiguous()

    def moe(c):
        vw4.verify_moe_w4(vw4.FMT_NVFP4, *gu[c], E, A, 0, ids_d, gates_d, 0, out=pair,
                          workspace=ws, stream=stream)
        vw4.verify_moe_w4(vw4.FMT_NVFP4, *dn[c], E, h, 1, ids_d, gates_d, 1, out=res,
                          workspace=ws, stream=stream)

    def timed(fn, reps):
        """Microseconds per fn call: a CUDA graph of fn(0), fn(1) (the two
        weight copies), replayed reps times (no host work in the timed loop)."""
        for c in range(4):
            fn(c % 2)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn(0)
            fn(1)
        with torch.cuda.stream(stream):  # replays and events on one stream
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (2 * reps) * 1e3

    us = timed(moe, 20)
    n_exp = len(set(int(x) for x in ids.reshape(-1)))
    moe_bytes = n_exp * (2 * f * d + d * f) * 9 // 16 + (M * d + M * topk * f) * 2
    out["moe_head_m8"] = {"us": round(us, 2), "distinct_experts": n_exp,
                          "gbs": round(moe_bytes / (us * 1e-6) / 1e9, 1)}
    # the same head with 16 tokens (128 routed pairs)
    M16 = 16
    ids16, gates16 = synth.routing(302, M16, E, topk)
    ids16_d = torch.from_numpy(np.ascontiguousarray(ids16, np.int32)).to(device)
    gates16_d = torch.from_numpy(np.ascontiguousarray(gates16, np.float32)).to(device)
    A16 = torch.from_numpy(synth.activations(synth.rng(303), M16, d).view(np.int16)).view(
        torch.bfloat16).to(device)
    pair16 = torch.empty((M16 * topk, 2 * f), dtype=torch.float32, device=device)
    res16 = torch.empty((M16, d), dtype=torch.float32, device=device)
    vw4.verify_moe_w4(vw4.FMT_NVFP4, *gu[0], E, A16, 0, ids16_d, gates16_d, 0, out=pair16,
                      workspace=ws, stream=stream)
    h16 = (torch.nn.functional.silu(pair16[:, :f]) * pair16[:, f:]).to(torch.bfloat16).contiguous()

    def moe16(c):
        vw4.verify_moe_w4(vw4.FMT_NVFP4, *gu[c], E, A16, 0, ids16_d, gates16_d, 0, out=pair16,
                          workspace=ws, stream=stream)
        vw4.verify_moe_w4(vw4.FMT_NVFP4, *dn[c], E, h16, 1, ids16_d, gates16_d, 1, out=res16,
                          workspace=ws, stream=stream)

    us = timed(moe16, 20)
    n_exp16 = len(set(int(x) for x in ids16.reshape(-1)))
    moe_bytes16 = n_exp16 * (2 * f * d + d * f) * 9 // 16 + (M16 * d + M16 * topk * f) * 2
    out["moe_head_m16"] = {"us": round(us, 2), "distinct_experts": n_exp16,
                           "gbs": round(moe_bytes16 / (us * 1e-6) / 1e9, 1)}
    del gu, dn, pair, res, h, pair16, res16, h16
    torch.cuda.empty_cache()

    V, K = 262144, 5376
    heads = [synth.linear(220 + c, V, K, "nvfp4") for c in range(2)]
    heads = [(torch.from_numpy(q).to(device), torch.from_numpy(sc).to(device), ts)
             for q, sc, ts in heads]
    Ah = torch.from_numpy(synth.activations(synth.rng(222), 8, K).view(np.int16)).view(
        torch.bfloat16).to(device)
    logits = torch.empty((8, V), dtype=torch.float32, device=device)
    am = torch.empty((8,), dtype=torch.int32, device=device)
    vw4.verify_gemm_w4(vw4.FMT_NVFP4, *heads[0], Ah, out=logits, row_argmax=am, workspace=ws,
                       stream=stream)
    torch.cuda.synchronize()
    drafts = am[:7].clone().reshape(1, 7)   # every draft agrees: the whole run commits
    tokens = torch.empty((1, 8), dtype=torch.int32, device=device)
    length = torch.empty((1,), dtype=torch.int32, device=device)

    def head(c):
        vw4.verify_gemm_w4(vw4.FMT_NVFP4, *heads[c], Ah, out=logits, row_argmax=am,
                           workspace=ws, stream=stream)
        vw4.accept_greedy(None, drafts, target_argmax=am, B=1, V=V, tokens=tokens,
                          length=length, stream=stream)

    hb = weight_bytes(V, K) + 8 * K * 2
    us = timed(head, 10)
    out["lmhead_fused_greedy_m8_two_launches"] = {
        "us": round(us, 2), "gbs": round(hb / (us * 1e-6) / 1e9, 1),
        "what": "verify_gemm_w4 (logits + fused argmax) then accept_greedy"}

    def head1(c):  # GEMM, argmax and accept in one launch, no logits written
        vw4.verify_greedy_w4(vw4.FMT_NVFP4, *heads[c], Ah, drafts, tokens=tokens, length=length,
                             workspace=ws, stream=stream)

    us = timed(head1, 10)
    out["lmhead_fused_greedy_m8"] = {"us": round(us, 2), "gbs": round(hb / (us * 1e-6) / 1e9, 1),
                                     "what": "verify_greedy_w4: one launch, no logits written"}

    # the LM head alone at each verify width (logits written, two weight
    # copies alternating: 1.58 GB, far above L2)
    lm_per_m = {}
    Ahs = {M: torch.from_numpy(synth.activations(synth.rng(230 + M), M, K).view(np.int16)).view(
        torch.bfloat16).to(device) for M in PER_M}
    lgs = {M: torch.empty((M, V), dtype=torch.float32, device=device) for M in PER_M}
    for M in PER_M:
        def lm(c, M=M):
            vw4.verify_gemm_w4(vw4.FMT_NVFP4, *heads[c], Ahs[M], out=lgs[M], workspace=ws,
                               stream=stream)
        us = timed(lm, 10)
        b = weight_bytes(V, K) + M * K * 2
        lm_per_m[str(M)] = {"us": round(us, 2), "gbs": round(b / (us * 1e-6) / 1e9, 1)}
    out["lmhead_per_m"] = lm_per_m
    del lgs

    # the sampled accept fed by the LM-head GEMM (B = 1 sequence, 7 drafts,
    # T = 0.6, top_p = 0.95): the verify GEMM's 8 rows, then the rejection
    # accept against the 7 draft rows (made once, by the same head, as a
    # drafter sharing it would).  Unfused: verify_gemm_w4 + accept_rejection;
    # fused: verify_gemm_w4_blockmax (logits and the maximum of every 16) +
    # accept_rejection_blockmax (no pass over the rows for their maxima).
    Kd = 7
    Ad7 = torch.from_numpy(synth.activations(synth.rng(240), Kd, K).view(np.int16)).view(
        torch.bfloat16).to(device)
    dlog, dbm = vw4.verify_gemm_w4_blockmax(vw4.FMT_NVFP4, *heads[0], Ad7, workspace=ws,
                                            stream=stream)
    torch.cuda.synchronize()
    g7 = torch.Generator(device=device).manual_seed(5)
    sd_drafts = torch.multinomial(torch.softmax(dlog / 0.6, dim=-1), 1, generator=g7).reshape(
        1, Kd).to(torch.int32)
    tlog = torch.empty((Kd + 1, V), dtype=torch.float32, device=device)
    tbm = torch.empty((Kd + 1, (V + 15) // 16), dtype=torch.float32, device=device)
    ws_acc = vw4.Workspace(device)
    tok_s = torch.empty((1, Kd + 1), dtype=torch.int32, device=device)
    len_s = torch.empty((1,), dtype=torch.int32, device=device)

    def sampled(c):
        vw4.verify_gemm_w4(vw4.FMT_NVFP4, *heads[c], Ah, out=tlog, workspace=ws, stream=stream)
        vw4.accept_rejection(tlog.view(1, Kd + 1, V), dlog.view(1, Kd, V), sd_drafts, 0.6, 0.95, 4,
                             c, tokens=tok_s, length=len_s, workspace=ws_acc, stream=stream)

    def sampled_fused(c):
        vw4.verify_gemm_w4_blockmax(vw4.FMT_NVFP4, *heads[c], Ah, out=tlog, block_max=tbm,
                                    workspace=ws, stream=stream)
        vw4.accept_rejection_blockmax(tlog.view(1, Kd + 1, V), tbm, dlog.view(1, Kd, V), dbm,
                                      sd_drafts, 0.6, 0.95, 4, c, tokens=tok_s, length=len_s,
                                      workspace=ws_acc, stream=stream)

    def accept_only(c):
        vw4.accept_rejection(tlog.view(1, Kd + 1, V), dlog.view(1, Kd, V), sd_drafts, 0.6, 0.95, 4,
                             c, tokens=tok_s, length=len_s, workspace=ws_acc, stream=stream)

    def accept_only_fused(c):
        vw4.accept_rejection_blockmax(tlog.view(1, Kd + 1, V), tbm, dlog.view(1, Kd, V), dbm,
                                      sd_drafts, 0.6, 0.95, 4, c, tokens=tok_s, length=len_s,
                                      workspace=ws_acc, stream=stream)

    us_u = timed(sampled, 10)
    us_f = timed(sampled_fused, 10)
    us_a = timed(accept_only, 10)
    us_af = timed(accept_only_fused, 10)
    out["lmhead_sampled_accept_m8"] = {
        "unfused_us": round(us_u, 2), "fused_us": round(us_f, 2),
        "accept_alone_us": round(us_a, 2), "accept_alone_fused_us": round(us_af, 2),
        "what": "B=1, 7 drafts, V=262144, T=0.6, top_p=0.95: verify_gemm_w4 + accept_rejection "
                "vs verify_gemm_w4_blockmax + accept_rejection_blockmax"}
    del heads, logits, tlog, dlog
    torch.cuda.empty_cache()
    return out


def run_e2e(vw4, layer, layer_b, device, steps, warmup, world):
    """Same step through the public API with pinned host inputs and outputs:
    every step copies its four activation inputs in and its four fp32
    results out.  As an engine would issue it, the step is part of a CUDA
    graph: the inputs, which sit contiguous in one pinned buffer, come in
    with one copy on a copy stream that the first GEMM waits for; the
    results of the first three GEMMs (contiguous too) go out with one copy
    on a second copy stream while the last GEMM runs, and the last result
    with one copy after it.  As in the headline, consecutive steps alternate
    two weight copies of the layer (so that nothing is served from L2) and
    are captured two to a graph."""
    import torch
    import synth
    stream = torch.cuda.Stream(device)  # graphs are captured off the default stream
    M = HEAD_M
    g = np.random.default_rng(11)
    Ks = [K for _, N, K, *_ in layer]
    Ns = [N for _, N, *_ in layer]
    in_off = np.cumsum([0] + [M * K for K in Ks]).tolist()
    out_off = np.cumsum([0] + [M * N for N in Ns]).tolist()
    host_in = torch.empty(in_off[-1], dtype=torch.bfloat16).pin_memory()
    for j, K in enumerate(Ks):
        bits = synth.activations(g, M, K)
        host_in[in_off[j]:in_off[j + 1]].copy_(
            torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(-1))
    host_out = torch.empty(out_off[-1], dtype=torch.float32).pin_memory()
    dev_in = torch.empty(in_off[-1], dtype=torch.bfloat16, device=device)
    dev_out = torch.empty(out_off[-1], dtype=torch.float32, device=device)
    d_in = [dev_in[in_off[j]:in_off[j + 1]].view(M, Ks[j]) for j in range(len(Ks))]
    d_out = [dev_out[out_off[j]:out_off[j + 1]].view(M, Ns[j]) for j in range(len(Ns))]
    last = len(Ns) - 1
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in, ev_head, ev_last = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()

    def make_step(lay):
        gemms = [vw4.PreparedGemm(vw4.FMT_NVFP4, qd, sd, ts, M, stream=stream)
                 for (name, N, K, qd, sd, ts) in lay]

        def step():
            s_in.wait_stream(stream)
            with torch.cuda.stream(s_in):
                dev_in.copy_(host_in, non_blocking=True)
                ev_in.record(s_in)
            stream.wait_event(ev_in)
            for j in range(len(lay)):
                gemms[j](d_in[j], d_out[j])  # on `stream`
                if j == last - 1:            # results 0 .. last-1 out, behind the last GEMM
                    ev_head.record(stream)
                    s_out.wait_event(ev_head)
                    with torch.cuda.stream(s_out):
                        host_out[:out_off[last]].copy_(dev_out[:out_off[last]],
                                                       non_blocking=True)
            ev_last.record(stream)
            s_out.wait_event(ev_last)
            with torch.cuda.stream(s_out):
                host_out[out_off[last]:].copy_(dev_out[out_off[last]:], non_blocking=True)
            stream.wait_stream(s_out)
        return step

    steps_ab = [make_step(layer), make_step(layer_b)]
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 2)):
            steps_ab[i % 2]()
    torch.cuda.synchronize()

    def capture(fn):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn()
        torch.cuda.synchronize()
        return gr

    def two():
        steps_ab[0]()
        steps_ab[1]()
    g_pair, g_one = capture(two), capture(steps_ab[0])
    with torch.cuda.stream(stream):  # replays run on the current stream: this one
        for _ in range((warmup + 1) // 2):
            g_pair.replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps // 2):
            g_pair.replay()
        if steps % 2:
            g_one.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = reduce_max(e0.elapsed_time(e1), world)
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out.numel() * host_out.element_size()
    value = step_bytes(M) * steps * world / (ms * 1e-3) / 1e9
    return {"value": round(value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h}


# ------------------------------------------------------- CPU oracle timing
class OracleWorkload:
    """The same packed layer for the CPU oracle: its four nvfp4 matrices generated
    once; a "sample" is a random subset of output rows of every linear."""

    def __init__(self):
        import oracle
        import synth
        oracle.build()
        self.lin = [synth.linear(100 + i, N, K, "nvfp4") for i, (_, N, K) in enumerate(STEP)]
        g = synth.rng(11)
        self.acts = [synth.activations(g, HEAD_M, K) for _, N, K in STEP]

    def run(self, frac: float, seed: int):
        """Returns (GB/s over the sampled algorithmic bytes, rows, seconds)."""
        import oracle
        g = np.random.default_rng(seed)
        rows, secs, nbytes = 0, 0.0, 0
        for (name, N, K), (q, s, ts), A in zip(STEP, self.lin, self.acts):
            n = max(1, int(round(N * frac)))
            cols = np.sort(g.choice(N, n, replace=False)).astype(np.int32)
            t = time.perf_counter()
            oracle.gemm_w4(oracle.FMT_NVFP4, N, K, q, s, ts, A, cols=cols)
            secs += time.perf_counter() - t
            rows += n
            nbytes += weight_bytes(n, K) + HEAD_M * K * 2
        return nbytes / secs / 1e9, rows, secs

    def frac_for(self, budget_s: float) -> float:
        """Sample fraction whose oracle time is about budget_s (one calibration
        run); above 1.0 the whole layer is run that many times."""
        _, _, secs = self.run(0.01, 1)
        return 0.01 * budget_s / max(secs, 1e-6)

    def run_budget(self, frac: float, seed: int):
        """run() over a fraction of the rows, or the whole layer repeated when
        frac > 1; returns (GB/s, rows, seconds)."""
        if frac <= 1.0:
            return self.run(frac, seed)
        reps = max(1, int(round(frac)))
        tot_rows, tot_s, gbs = 0, 0.0, []
        for r in range(reps):
            v, rows, secs = self.run(1.0, seed + r)
            gbs.append(v)
            tot_rows += rows
            tot_s += secs
        return len(gbs) / sum(1.0 / v for v in gbs), tot_rows, tot_s


def cpu_cores():
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def reduce_max(value: float, world: int) -> float:
    """Max of a per-rank float over all ranks (identity for one process)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on this machine's host cores,
    each step a bounded sample of the same workload.  Rank 0 only."""
    if rank != 0:
        return None
    wl = OracleWorkload()
    per_step_budget = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    frac = wl.frac_for(per_step_budget)
    for k in range(args.warmup):
        wl.run_budget(frac, 1000 + k)
    vals, rows = [], 0
    t0 = time.perf_counter()
    for k in range(args.steps):
        v, rows, _ = wl.run_budget(frac, 2000 + k)
        vals.append(v)
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    what = (f"a {frac:.4%} random subset of the output rows of the layer's 4 packed matrices" if frac <= 1.0
            else f"the whole packed layer, {int(round(frac))} times")
    sample = f"each step: {what} ({rows} rows), M=8, nvfp4; fp64 dequantize-and-dot"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": HEAD_M, "fmt": "nvfp4"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_case(case: str, device):
    """Profiling helper: a few calls of the GEMM on a fixed case, nothing timed
    or printed but a one-line summary.  'dense' = the 4 nvfp4 calls of the
    packed layer step at M = 8 (3 warm-up passes, then 1); 'N,K,M[,q4_0]' = one
    GEMM of that shape, nvfp4 unless q4_0 is named (3 warm-up calls, then 1); 'rejection:K' = the
    rejection accept of the stochastic sweep (B = 256, V = 151936, K drafts),
    4 calls; 'lists:K' = the accept over top-64 lists of those rows, 4 calls;
    'moe:M' = the MoE head (gate/up, then down with the gate combine) at M
    tokens, 4 calls; 'sampled:K' = one sequence's rejection accept with K
    drafts over 262144-entry rows of the LM head's logit spread, 4 calls."""
    import torch
    import speculative_decode_verification_w4_gb300 as vw4
    torch.cuda.set_device(device)
    ws = vw4.Workspace(device)
    if case.startswith("rejection:"):  # the stochastic sweep's accept step, K drafts
        Kd, B, V = int(case.split(":")[1]), 256, 151936
        g = torch.Generator(device=device).manual_seed(4)
        tgt = torch.randn((B, Kd + 1, V), generator=g, device=device) * 3.0
        drf = tgt[:, :Kd] + torch.randn((B, Kd, V), generator=g, device=device)
        probs = torch.softmax(drf.reshape(-1, V) / 0.6, dim=-1)
        drafts = torch.multinomial(probs, 1, generator=g).reshape(B, Kd).to(torch.int32)
        del probs
        for r in range(4):
            tok, ln = vw4.accept_rejection(tgt, drf, drafts, 0.6, 0.95, 4, r, workspace=ws)
        torch.cuda.synchronize()
        print(f"case {case}: 4 calls, mean run {ln.float().mean().item():.3f}, device status "
              f"{vw4.vw4_get_device_status()}", flush=True)
        return
    if case.startswith("lists:"):  # the accept over top-64 lists of the sweep rows, K drafts
        Kd, B, V, Kt = int(case.split(":")[1]), 256, 151936, 64
        g = torch.Generator(device=device).manual_seed(4)
        tgt = torch.randn((B, Kd + 1, V), generator=g, device=device) * 3.0
        drf = tgt[:, :Kd] + torch.randn((B, Kd, V), generator=g, device=device)
        tv, ti = torch.topk(tgt, Kt, dim=-1)
        dv, di = torch.topk(drf, Kt, dim=-1)
        ti, di = ti.to(torch.int32).contiguous(), di.to(torch.int32).contiguous()
        tv, dv = tv.contiguous(), dv.contiguous()
        del tgt, drf
        pick = torch.multinomial(torch.softmax(dv.reshape(-1, Kt) / 0.6, dim=-1), 1,
                                 generator=g).reshape(B, Kd, 1)
        ldrafts = torch.gather(di, 2, pick).reshape(B, Kd).contiguous()
        for r in range(4):
            tok, ln = vw4.accept_rejection_topk(ti, tv, di, dv, ldrafts, V, 0.6, 0.95, 4, r,
                                                workspace=ws)
        torch.cuda.synchronize()
        print(f"case {case}: 4 calls, mean run {ln.float().mean().item():.3f}, device status "
              f"{vw4.vw4_get_device_status()}", flush=True)
        return
    if case.startswith("sampled:"):  # one sequence's rejection accept at the LM head's width
        Kd, V = int(case.split(":")[1]), 262144
        g = torch.Generator(device=device).manual_seed(5)
        # logits of the LM head's spread: N(0, 0.02^2 * 5376) per entry
        tgt = torch.randn((1, Kd + 1, V), generator=g, device=device) * 1.466
        drf = torch.randn((1, Kd, V), generator=g, device=device) * 1.466
        drafts = torch.multinomial(torch.softmax(drf.reshape(-1, V) / 0.6, dim=-1), 1,
                                   generator=g).reshape(1, Kd).to(torch.int32)
        for r in range(4):
            tok, ln = vw4.accept_rejection(tgt, drf, drafts, 0.6, 0.95, 4, r, workspace=ws)
        torch.cuda.synchronize()
        print(f"case {case}: 4 calls, run {ln.item()}, device status "
              f"{vw4.vw4_get_device_status()}", flush=True)
        return
    if case.startswith("moe:"):  # the MoE head (gate/up then down with the combine), M tokens
        import synth
        M = int(case.split(":")[1])
        E, d, f, topk = 128, 2048, 768, 8
        gu = [torch.from_numpy(x).to(device) if isinstance(x, np.ndarray) else x
              for x in synth.linear(200, E * 2 * f, d, "nvfp4")]
        dn = [torch.from_numpy(x).to(device) if isinstance(x, np.ndarray) else x
              for x in synth.linear(210, E * d, f, "nvfp4")]
        ids, gates = synth.routing(300 if M == 8 else 302, M, E, topk)
        ids_d = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).to(device)
        gates_d = torch.from_numpy(np.ascontiguousarray(gates, np.float32)).to(device)
        A = torch.from_numpy(synth.activations(synth.rng(301), M, d).view(np.int16)).view(
            torch.bfloat16).to(device)
        pair = torch.empty((M * topk, 2 * f), dtype=torch.float32, device=device)
        res = torch.empty((M, d), dtype=torch.float32, device=device)
        h = torch.zeros((M * topk, f), dtype=torch.bfloat16, device=device)
        for _ in range(4):
            vw4.verify_moe_w4(vw4.FMT_NVFP4, *gu, E, A, 0, ids_d, gates_d, 0, out=pair,
                              workspace=ws)
            vw4.verify_moe_w4(vw4.FMT_NVFP4, *dn, E, h, 1, ids_d, gates_d, 1, out=res,
                              workspace=ws)
        torch.cuda.synchronize()
        print(f"case {case}: 4 head calls, device status {vw4.vw4_get_device_status()}",
              flush=True)
        return
    if case == "dense":
        layer = make_layer("nvfp4", device)
        acts = make_acts(HEAD_M, device, seed=7 + HEAD_M)
        jobs = [(qd, sd, ts, acts[j], N) for j, (name, N, K, qd, sd, ts) in enumerate(layer)]
    else:
        import synth
        parts = case.split(",")
        N, K, M = (int(x) for x in parts[:3])
        fmt = parts[3] if len(parts) > 3 else "nvfp4"
        q, sc, ts = synth.linear(1, N, K, fmt)
        bits = synth.activations(synth.rng(2), M, K)
        A = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)
        sd = torch.from_numpy(sc if fmt == "nvfp4" else sc.view(np.uint16)).to(device)
        if fmt != "nvfp4":
            sd = sd.view(torch.float16)
        jobs = [(torch.from_numpy(q).to(device), sd, ts, A, N)]
    code = vw4.FMT_Q4_0 if case.endswith("q4_0") else vw4.FMT_NVFP4
    outs = [torch.empty((a.shape[0], N), dtype=torch.float32, device=device)
            for (_, _, _, a, N) in jobs]
    for _ in range(4):
        for (qd, sd, ts, a, N), o in zip(jobs, outs):
            vw4.verify_gemm_w4(code, qd, sd, ts, a, out=o, workspace=ws)
    torch.cuda.synchronize()
    print(f"case {case}: {len(jobs)} GEMM(s) x 4 calls, device status "
          f"{vw4.vw4_get_device_status()}", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--case", default=None,
                    help="profiling helper: 'dense', 'N,K,M[,q4_0]', 'rejection:K', 'lists:K', 'moe:M' or 'sampled:K' (see run_case); "
                         "no JSON line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    import torch
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    if args.case:
        run_case(args.case, device)
        return
    res = run_ours(args, rank, world, device)
    if rank == 0:
        wl = OracleWorkload()
        frac = wl.frac_for(args.cpu_budget)
        v, rows, secs = wl.run_budget(frac, 7)
        what = (f"{frac:.4%} of the output rows of the layer's 4 packed matrices" if frac <= 1.0
                else f"the whole packed layer, {int(round(frac))} times")
        res["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cpu_cores(),
                               "kind": "oracle",
                               "sample": f"{what} ({rows} rows, {secs:.1f} s), M=8, nvfp4, "
                                         f"fp64 dequantize-and-dot"}
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
