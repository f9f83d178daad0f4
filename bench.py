#!/usr/bin/env python3
"""Benchmark of the F16-weight products on one GB300 (or N replicas).

Default workload (the JSON line's `value`): a Llama-3-8B-shaped decode step --
32 layers of [fused Q/K/V product (4096+1024+1024 rows x 4096), O (4096 x 4096),
fused gate/up (2 x 14336 x 4096), down (4096 x 14336)] then the output product
(128256 x 4096): one column, 129 products over 15.0 GB of f16 weights (far more
than the 129 MB L2), seeded synthetic weights N(0, 0.01) (one layer drawn and
copied to 32 distinct buffers, so every product streams from HBM) and a distinct
f32 activation N(0, 1) for every product.  Each product is one
bm_f16_matvec_act call: the f32 activation is rounded to f16 and multiplied in
the same launch (k_gemv_stream).  The step is captured once as a CUDA graph
(programmatic dependent launch on) and replayed; `value` is algorithmic bytes
per step / time per step.

Objects in the same JSON line:
  roofline     -- the step's only kernel (k_gemv_stream) against the measured HBM peak,
                  with the DRAM traffic per launch from an ncu launch list
  e2e          -- the same step end to end: every step the activations are copied
                  from pinned host memory, the 129 recorded calls are made one C call
                  each, the logits are copied back and the host waits for them
  cpu_baseline -- the CPU oracle on this host, on a bounded sample of the same step
  prefill      -- the second half of the metric: one Llama-3-8B-shaped layer's
                  products for a 512-token prefill micro-batch on the tensor cores,
                  TFLOP/s against the measured dense bf16 peak
  smollm2_135m_decode_step, qwen3_0.6b_decode_step -- the smaller decode steps
                  (launch-latency-bound), with their unfused and norm-fused variants
  products     -- single products: one and few columns (HBM GB/s), 512 columns
                  (TFLOP/s), and the exact fallback and unaligned shapes
  helpers      -- rms_norm_mul, get_rows, mad and scale

`--impl reference` times the CPU oracle (the only reference that exists for
this method) on the same workload and metric, on a bounded sample of the step.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

SEED = 0
A_SIGMA = 1.0

# The decode steps' shapes.  distinct: every layer's weights drawn on their own
# (else one layer is drawn and copied to every layer's buffers).
MODELS = {
    "smollm2_135m": {"prefix": "smollm2", "hidden": 576, "q": 9 * 64, "kv": 3 * 64, "o_in": 576, "ffn": 1536,
                     "vocab": 49152, "head": "token_embd", "layers": 30, "sigma": 0.02, "distinct": True},
    "qwen3_0.6b": {"prefix": "qwen3", "hidden": 1024, "q": 16 * 128, "kv": 8 * 128, "o_in": 16 * 128, "ffn": 3072,
                   "vocab": 151936, "head": "embd", "layers": 28, "sigma": 0.02, "distinct": False},
    "llama3_8b": {"prefix": "llama3_8b", "hidden": 4096, "q": 32 * 128, "kv": 8 * 128, "o_in": 32 * 128,
                  "ffn": 14336, "vocab": 128256, "head": "output", "layers": 32, "sigma": 0.01, "distinct": False},
}
HEADLINE = "llama3_8b"


def weight_name(model: str, layer: int, mat: str) -> str:
    m = MODELS[model]
    if mat == "head":
        return "%s.%s" % (m["prefix"], m["head"])
    return "%s.l%d.%s" % (m["prefix"], layer, mat) if m["distinct"] else "%s.%s" % (m["prefix"], mat)


def step_plan(model: str = HEADLINE, layers: int | None = None):
    """The decode step as an ordered list of calls (kind, [(output key, weight name,
    rows)], k, activation id); kind is 'multi' (one launch over several matrices),
    'mv' or 'logits'.  Every call has its own activation."""
    m = MODELS[model]
    L = m["layers"] if layers is None else layers
    h, plan, a = m["hidden"], [], 0
    for i in range(L):
        def mats(*names):
            return [("l%d.%s" % (i, n), weight_name(model, i, n), r) for n, r in names]
        plan.append(("multi", mats(("q", m["q"]), ("k", m["kv"]), ("v", m["kv"])), h, a))
        plan.append(("mv", mats(("o", h)), m["o_in"], a + 1))
        plan.append(("multi", mats(("gate", m["ffn"]), ("up", m["ffn"])), h, a + 2))
        plan.append(("mv", mats(("down", h)), m["ffn"], a + 3))
        a += 4
    plan.append(("logits", [("head", weight_name(model, 0, "head"), m["vocab"])], h, a))
    return plan


def act_name(model: str, a: int) -> str:
    return "%s.act%d" % (MODELS[model]["prefix"], a)


def step_bytes(plan, fused=True):
    """Algorithmic bytes of one step.  Fused: each call reads its f32 activation (4k)
    and rounds it in the kernel; unfused: a rounding call (6 bytes per element), then
    the product reads the f16 activation (2k).  Weights 2*rows*k and outputs 4*rows
    either way; a multi-matrix call reads its activation once."""
    tot = 0
    for _, mats, k, _ in plan:
        tot += sum(2 * r * k + 4 * r for _, _, r in mats) + (4 * k if fused else 6 * k + 2 * k)
    return tot


def weight_bytes(plan):
    return sum(2 * r * k for _, mats, k, _ in plan for _, _, r in mats)


def algorithmic_bytes(rows, k, ncols=1):
    return 2 * rows * k + 2 * k * ncols + 4 * rows * ncols


# DRAM traffic of k_gemv_stream per product shape (rows x k, matrices of one launch),
# from the ncu launch list of a two-layer Llama-3-8B-shaped step (read + write bytes,
# profiles/decode_step_llama3_8b_launches.md), valid only for the kernel source it was
# measured on (sha256 prefix of k_gemv_stream.cu).  Shapes per launch do not depend on
# the number of layers, so the full step's traffic is these, summed over its launches.
NCU_TRAFFIC = {"kernel": "k_gemv_stream", "source": "f16_weight_gemv_gb300/csrc/k_gemv_stream.cu",
               "sha256_16": "ab91cb641fe613cf",
               "bytes_per_call": {"4096x4096+1024x4096+1024x4096": 50420864, "4096x4096": 33638912,
                                  "14336x4096+14336x4096": 235086592, "4096x14336": 117655552,
                                  "128256x4096": 1051435264}}


# DRAM traffic of the prefill layer's four k_gemm_tc launches (Q/K/V, O, gate/up, down; read +
# write bytes), from the ncu launch list in profiles/prefill_layer_llama3_8b_launches.md, valid
# only for the kernel source it was measured on.
PREFILL_TRAFFIC = {"kernel": "k_gemm_tc", "source": "f16_weight_gemv_gb300/csrc/k_gemm_tc.cu",
                   "sha256_16": "c52fe893d3def690", "bytes_per_launch": [54795264, 37834496, 281310976, 132292096]}


def prefill_traffic_per_launch():
    t = PREFILL_TRAFFIC
    if not t["sha256_16"] or _source_sha16(t["source"]) != t["sha256_16"]:
        return None
    return int(round(sum(t["bytes_per_launch"]) / len(t["bytes_per_launch"])))


def _source_sha16(rel):
    import hashlib
    try:
        with open(os.path.join(ROOT, rel), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None


def call_key(mats, k):
    return "+".join("%dx%d" % (r, k) for _, _, r in mats)


def ncu_traffic_per_launch(plan):
    """Mean DRAM bytes per launch of the step from the recorded per-shape traffic, or
    None when the kernel changed since (or a shape was not measured)."""
    t = NCU_TRAFFIC
    if not t["sha256_16"] or _source_sha16(t["source"]) != t["sha256_16"]:
        return None
    tot = 0
    for _, mats, k, _ in plan:
        b = t["bytes_per_call"].get(call_key(mats, k))
        if b is None:
            return None
        tot += b
    return int(round(tot / len(plan)))


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "25"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.03 <= r[0] <= t1 + 0.03]
        if len(inside) < 3:  # a short timed region: the samples nearest to it
            inside = sorted(rows, key=lambda r: abs(r[0] - 0.5 * (t0 + t1)))[:3]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower() not in ("not active", "0x0000000000000000", "0", "[n/a]", "n/a"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# ----------------------------------------------------------------------------- decode steps


class DecodeStep:
    """A decode step of `model` resident on the GPU: weights, one f32 activation per
    call (packed, 32-byte aligned slices), one output per matrix and layer.  With
    keep_host the host copies of the distinct weights and of the activations stay
    (for the parity tests)."""

    def __init__(self, bm, torch, dev, model=HEADLINE, layers=None, keep_host=False):
        self.bm, self.torch, self.model = bm, torch, model
        spec = MODELS[model]
        self.plan = step_plan(model, layers)
        self.host_w = {}
        dev_by_name = {}
        for _, mats, k, _ in self.plan:
            for _, wn, rows in mats:
                if wn in dev_by_name:
                    continue
                w = synth.normal_f16(SEED, wn, spec["sigma"], (rows, k))
                dev_by_name[wn] = torch.from_numpy(w.view(np.float16)).to(dev)
                if keep_host:
                    self.host_w[wn] = w
        # one layer drawn: every layer gets its own copy (distinct memory, streamed from HBM)
        self.weights = {}
        for _, mats, _, _ in self.plan:
            for key, wn, _ in mats:
                layer0 = key.startswith("l0.") or key == "head" or spec["distinct"]
                self.weights[key] = dev_by_name[wn] if layer0 else dev_by_name[wn].clone()
        del dev_by_name
        self.offs, o = {}, 0
        for _, _, k, a in self.plan:
            self.offs[a] = (o, k)
            o += (k + 7) // 8 * 8
        self.act_host = np.zeros(o, dtype=np.float32)
        for a, (off, k) in self.offs.items():
            self.act_host[off:off + k] = synth.normal_f32(SEED, act_name(model, a), A_SIGMA, k)
        self.act = torch.from_numpy(self.act_host).to(dev)
        self.act_f16 = None
        self.outs = {key: torch.empty(rows, dtype=torch.float32, device=dev)
                     for _, mats, _, _ in self.plan for key, _, rows in mats}
        self.norm_w = torch.from_numpy((1.0 + synth.normal_f32(SEED, "%s.norm" % spec["prefix"], 0.2,
                                                               spec["hidden"])).astype(np.float32)).to(dev)
        self.bytes = step_bytes(self.plan, True)

    def activation(self, a):
        off, k = self.offs[a]
        return self.act[off:off + k]

    def run(self, s, mode="act"):
        """mode 'act': one bm_f16_matvec_act per call (the benchmarked step); 'unfused':
        bm_to_f16, then bm_f16_matvec[_multi] / bm_f16_logits; 'norm': the RMS norm fused
        ahead of Q/K/V, gate/up and the head (bm_f16_matvec_norm)."""
        bm = self.bm
        if mode == "unfused" and self.act_f16 is None:
            self.act_f16 = self.torch.empty(self.act.numel(), dtype=self.torch.float16, device=self.act.device)
        for kind, mats, k, a in self.plan:
            W = [self.weights[key] for key, _, _ in mats]
            Y = [self.outs[key] for key, _, _ in mats]
            x = self.activation(a)
            if mode == "act" or (mode == "norm" and kind == "mv"):
                bm.bm_f16_matvec_act(W, x, Y, stream=s)
            elif mode == "norm":
                bm.bm_f16_matvec_norm(W, x, self.norm_w, 1e-5, Y, stream=s)
            else:
                off, _ = self.offs[a]
                h = self.act_f16[off:off + k]
                bm.bm_to_f16(x, h, stream=s)
                if kind == "multi":
                    bm.bm_f16_matvec_multi(W, h, Y, stream=s)
                elif kind == "mv":
                    bm.bm_f16_matvec(W[0], h, Y[0], stream=s)
                else:
                    bm.bm_f16_logits(W[0], h.view(1, -1), Y[0].view(1, -1), stream=s)

    def record(self):
        """The step's calls recorded as one launch (bm_step_create): the same products, in
        the same order, with the same bits as run()."""
        return self.bm.bm_step_create([([self.weights[key] for key, _, _ in mats], self.activation(a),
                                        [self.outs[key] for key, _, _ in mats]) for _, mats, _, a in self.plan])

    def head(self):
        return self.outs["head"]


def capture(torch, stream, fn):
    """fn() once eagerly (attribute set-up happens outside capture), then captured."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def replay_time(torch, stream, g, steps, warmup, world=1):
    """ms per replay of graph g: `warmup` untimed replays, then `steps` between CUDA
    events on the launching stream, a barrier and a synchronize on both sides."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    return e0.elapsed_time(e1) / steps


def e2e_time(torch, stream, step, calls, steps):
    """ms per step end to end: each step copies the step's activations from pinned host
    memory, makes the step's calls, copies the logits back and waits for them on the
    host (wall clock over `steps` such steps, after two untimed ones)."""
    act_pinned = torch.from_numpy(step.act_host).pin_memory()
    head_host = torch.empty(step.head().numel(), dtype=torch.float32).pin_memory()

    def one():
        with torch.cuda.stream(stream):
            step.act.copy_(act_pinned, non_blocking=True)
            calls()
            head_host.copy_(step.head(), non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    return (time.perf_counter() - t0) * 1e3 / steps, int(step.act_host.nbytes), int(head_host.numel() * 4)


def one_launch_time(torch, stream, st, steps, warmup=3):
    """ms per run of the step recorded as one launch (bm_step_create / bm_step_run):
    CUDA events on the launching stream around `steps` runs."""
    step = st.record()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step.run(stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step.run(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    step.close()
    return e0.elapsed_time(e1) / steps


def decode_side(bm, torch, dev, stream, model, steps=20, variants=True):
    """A smaller decode step as a side measurement: the fused step (as the headline),
    the same calls recorded as one launch, and optionally its unfused and norm-fused
    variants and its end-to-end time."""
    st = DecodeStep(bm, torch, dev, model)
    g = capture(torch, stream, lambda: st.run(stream))
    ms = replay_time(torch, stream, g, steps, 5)
    ms1 = one_launch_time(torch, stream, st, steps)
    res = {"ms_per_step": round(ms, 5), "GB_s": round(st.bytes / ms / 1e6, 1), "launches": len(st.plan),
           "weight_GB": round(weight_bytes(st.plan) / 1e9, 3),
           "how": "%d bm_f16_matvec_act calls (rounding fused), CUDA graph, PDL on" % len(st.plan),
           "one_launch": {"ms_per_step": round(ms1, 5), "GB_s": round(st.bytes / ms1 / 1e6, 1),
                          "how": "the same calls recorded once (bm_step_create) and run as one cooperative launch "
                                 "(bm_step_run), each call waiting on the device for every earlier call"}}
    if variants:
        g_u = capture(torch, stream, lambda: st.run(stream, "unfused"))
        ms_u = replay_time(torch, stream, g_u, steps, 5)
        unfused_bytes = step_bytes(st.plan, False)
        res["unfused"] = {"ms_per_step": round(ms_u, 5), "GB_s": round(unfused_bytes / ms_u / 1e6, 1),
                          "launches": 2 * len(st.plan),
                          "how": "bm_to_f16 then bm_f16_matvec[_multi] / bm_f16_logits per product"}
        g_n = capture(torch, stream, lambda: st.run(stream, "norm"))
        ms_n = replay_time(torch, stream, g_n, steps, 5)
        nb = st.bytes + 4 * MODELS[model]["hidden"] * sum(1 for op in st.plan if op[0] != "mv")
        res["norm_front_end"] = {"ms_per_step": round(ms_n, 5), "GB_s": round(nb / ms_n / 1e6, 1),
                                 "how": "the RMS norm ahead of Q/K/V, gate/up and the head fused into those "
                                        "launches (bm_f16_matvec_norm)"}
        prepared = bm.prepare(lambda: st.run(stream))
        ms_e, h2d, d2h = e2e_time(torch, stream, st, prepared, max(3, min(steps, 30)))
        res["e2e"] = {"GB_s": round(st.bytes / ms_e / 1e6, 1), "ms_per_step": round(ms_e, 5),
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "how": "recorded calls replayed one C call each; activations in, logits out, host waits"}
        del g_u, g_n
    del g, st
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- GPU arm


def run_gpu(args, rank, world, local_rank):
    import torch

    import f16_weight_gemv_gb300 as bm

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    bm.lib()
    stream = torch.cuda.Stream(device=dev)
    # The weights are constants: programmatic dependent launch lets each product start
    # copying its weights while the kernel ahead of it is still running.
    bm.bm_set_pdl(not args.no_pdl)

    step = DecodeStep(bm, torch, dev, HEADLINE, args.decode_layers)
    g_step = capture(torch, stream, lambda: step.run(stream))

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else
                          int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank]))
    clocks.start()
    time.sleep(0.3)
    t_begin = time.time()
    ms = replay_time(torch, stream, g_step, args.steps, args.warmup, world)
    t_end = time.time()
    time.sleep(0.1)
    clk = clocks.summary(t_begin, t_end)
    clocks.stop()
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())

    # ---- end to end through the binding: the step's 129 calls recorded once by prepare()
    # (arguments checked and marshalled once), then every step: activations in from pinned
    # host memory, one C call per product, logits out, the host waits for them
    e2e_steps = max(3, min(args.steps, 30))
    prepared = bm.prepare(lambda: step.run(stream))
    ms_e2e, h2d, d2h = e2e_time(torch, stream, step, prepared, e2e_steps)
    pg = prepared.graph(stream)
    ms_e2e_graph, _, _ = e2e_time(torch, stream, step, pg, e2e_steps)
    ms_e2e_eager, _, _ = e2e_time(torch, stream, step, lambda: step.run(stream), e2e_steps)
    del pg, prepared, g_step
    ms_one = one_launch_time(torch, stream, step, max(3, min(args.steps, 20)))

    result = {"ms": ms, "ms_e2e": ms_e2e, "ms_e2e_graph": ms_e2e_graph, "ms_e2e_eager": ms_e2e_eager, "ms_one": ms_one,
              "tot_bytes": step.bytes, "weight_bytes": weight_bytes(step.plan), "launches_per_step": len(step.plan),
              "plan": step.plan, "clocks": clk, "h2d": h2d, "d2h": d2h}
    del step
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_products:
        result["prefill"] = bench_llama_prefill(bm, dev, stream, torch)
        result["smollm2_135m_decode_step"] = decode_side(bm, torch, dev, stream, "smollm2_135m")
        result["qwen3_0.6b_decode_step"] = decode_side(bm, torch, dev, stream, "qwen3_0.6b", variants=False)
        result["qwen3_0.6b_prefill_layer"] = bench_qwen3_prefill(bm, dev, stream, torch)
        result["products"] = bench_products(bm, dev, stream, torch)
        result["helpers"] = bench_helpers(bm, dev, stream, torch)
    return result


def graph_time(torch, stream, fn, reps=3, pre=None):
    """Capture fn() once as a CUDA graph; median ms of `reps` replays (pre() runs
    before each replay, outside the timed events)."""
    g = capture(torch, stream, fn)
    ts = []
    for _ in range(reps):
        with torch.cuda.stream(stream):
            if pre is not None:
                pre()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return float(np.median(ts))


class PrefillLayer:
    """One Llama-3-8B-shaped layer's products for a prefill micro-batch of `n` tokens,
    resident on the GPU: Q/K/V/O (4096, 1024, 1024, 4096 rows x 4096), gate and up
    (14336 x 4096) and down (4096 x 14336), weights N(0, 0.01); the normed activations
    x (f32 [n][4096]) and the FFN activation xf (f32 [n][14336], a synthetic stand-in for
    the SwiGLU output) N(0, 1), each rounded to f16 by bm_to_f16 inside the step.  7
    tensor-core products and 2 rounding kernels per step (plus a reduction after each
    product that splits k).  The layer's 436 MB of weights exceed L2, so replays stream
    them from HBM."""

    HID, FFN, KV = 4096, 14336, 1024
    SHAPES = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096), ("gate", 14336, 4096),
              ("up", 14336, 4096), ("down", 4096, 14336)]

    def __init__(self, bm, torch, dev, n=512, keep_host=False):
        self.bm, self.torch, self.n = bm, torch, n
        self.host = {}
        self.W = {}
        for nm, r, c in self.SHAPES:
            w = synth.normal_f16(SEED, "llama3_8b." + nm, 0.01, (r, c))
            self.W[nm] = torch.from_numpy(w.view(np.float16)).to(dev)
            if keep_host:
                self.host[nm] = w
        xh = synth.normal_f32(SEED, "llama3_8b.prefill_x", 1.0, (n, self.HID))
        fh = synth.normal_f32(SEED, "llama3_8b.prefill_ffn", 1.0, (n, self.FFN))
        if keep_host:
            self.host["x"], self.host["xf"] = xh, fh
        self.x = torch.from_numpy(xh).to(dev)
        self.xf = torch.from_numpy(fh).to(dev)
        self.h = torch.empty((n, self.HID), dtype=torch.float16, device=dev)
        self.hd = torch.empty((n, self.FFN), dtype=torch.float16, device=dev)
        self.Y = {nm: torch.empty((n, r), dtype=torch.float32, device=dev) for nm, r, _ in self.SHAPES}
        self.flops = 2.0 * n * sum(r * c for _, r, c in self.SHAPES)
        self._cat = None

    def run(self, s, variant="multi"):
        """variant 'separate': 7 bm_f16_matmul calls; 'multi': Q/K/V and gate/up each one
        bm_f16_matmul_multi launch (the separate matrices share the activation); 'concat':
        Q/K/V and gate/up stored as one matrix each ([6144][4096] and [28672][4096]), whose
        outputs a caller reads as row ranges of each column."""
        bm, W, Y = self.bm, self.W, self.Y
        bm.bm_to_f16(self.x, self.h, stream=s)
        if variant == "separate":
            for nm in ("q", "k", "v", "o", "gate", "up"):
                bm.bm_f16_matmul(W[nm], self.h, Y=Y[nm], stream=s)
        elif variant == "multi":
            bm.bm_f16_matmul_multi([W["q"], W["k"], W["v"]], self.h, [Y["q"], Y["k"], Y["v"]], stream=s)
            bm.bm_f16_matmul(W["o"], self.h, Y=Y["o"], stream=s)
            bm.bm_f16_matmul_multi([W["gate"], W["up"]], self.h, [Y["gate"], Y["up"]], stream=s)
        else:
            if self._cat is None:
                t = self.torch
                Wqkv = t.cat([W["q"], W["k"], W["v"]], 0)
                Wgu = t.cat([W["gate"], W["up"]], 0)
                self._cat = (Wqkv, Wgu, t.empty((self.n, Wqkv.shape[0]), dtype=t.float32, device=Wqkv.device),
                             t.empty((self.n, Wgu.shape[0]), dtype=t.float32, device=Wqkv.device))
            Wqkv, Wgu, Yqkv, Ygu = self._cat
            bm.bm_f16_matmul(Wqkv, self.h, Y=Yqkv, stream=s)
            bm.bm_f16_matmul(W["o"], self.h, Y=Y["o"], stream=s)
            bm.bm_f16_matmul(Wgu, self.h, Y=Ygu, stream=s)
        bm.bm_to_f16(self.xf, self.hd, stream=s)
        bm.bm_f16_matmul(W["down"], self.hd, Y=Y["down"], stream=s)


def bench_llama_prefill(bm, dev, stream, torch, reps=10):
    """The prefill half of the metric: PrefillLayer at 512 tokens as one CUDA graph, with
    Q/K/V and gate/up through bm_f16_matmul_multi and programmatic dependent launch (the
    `value`), and the other variants beside it."""
    layer = PrefillLayer(bm, torch, dev)
    old = bm.bm_set_pdl(True)
    try:
        ms = graph_time(torch, stream, lambda: layer.run(stream, "multi"), reps=reps)
        ms_sep = graph_time(torch, stream, lambda: layer.run(stream, "separate"), reps=reps)
        ms_cat = graph_time(torch, stream, lambda: layer.run(stream, "concat"), reps=reps)
        bm.bm_set_pdl(False)
        ms_plain = graph_time(torch, stream, lambda: layer.run(stream, "multi"), reps=reps)
    finally:
        bm.bm_set_pdl(old)
    tf = lambda t: round(layer.flops / t / 1e9, 1)  # noqa: E731
    res = {"workload": "llama3_8b_prefill_layer", "tokens": layer.n, "ms_per_step": round(ms, 4),
           "TFLOP_s": tf(ms), "flop_per_step": layer.flops,
           "how": "one layer's 7 products at 512 columns (Q/K/V and gate/up through bm_f16_matmul_multi) plus 2 "
                  "rounding kernels, CUDA graph, PDL on; median of %d replays, weights (436 MB) larger than L2" % reps,
           "separate": {"ms_per_step": round(ms_sep, 4), "TFLOP_s": tf(ms_sep),
                        "how": "7 bm_f16_matmul calls, PDL on"},
           "concatenated_weights": {"ms_per_step": round(ms_cat, 4), "TFLOP_s": tf(ms_cat),
                                    "how": "Q/K/V and gate/up each stored as one matrix: 4 products, PDL on"},
           "without_pdl": {"ms_per_step": round(ms_plain, 4), "TFLOP_s": tf(ms_plain)}}
    # the products one by one (each a graph of one call after an L2 flush by a read)
    flush_buf = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sink = torch.zeros((), dtype=torch.float32, device=dev)
    per = []
    for nm, r, c in PrefillLayer.SHAPES:
        X = layer.hd if nm == "down" else layer.h
        t = graph_time(torch, stream, lambda: bm.bm_f16_matmul(layer.W[nm], X, Y=layer.Y[nm], stream=stream),
                       reps=5, pre=lambda: sink.copy_(flush_buf.sum()))
        per.append({"product": nm, "rows": r, "k": c, "us": round(t * 1e3, 2),
                    "TFLOP_s": round(2.0 * r * c * layer.n / t / 1e9, 1), "plan": bm.bm_tc_plan(r, c, layer.n)})
    res["products"] = per
    del layer, flush_buf
    torch.cuda.empty_cache()
    return res


def bench_qwen3_prefill(bm, dev, stream, torch, reps=10):
    """A Qwen3-0.6B-shaped prefill micro-batch of 512 tokens through one layer's products,
    with Q/K/V and gate/up stored as one matrix each ([4096][1024] and [6144][1024]), then
    O (1024 x 2048) and down (1024 x 3072), plus the two roundings: one CUDA graph, PDL on.
    One layer's weights (31 MB) sit in L2, so this measures the tensor path with hot weights."""
    hid, q, kv, ffn, n = 1024, 2048, 1024, 3072, 512
    Wqkv = torch.from_numpy(synth.normal_f16(SEED, "qwen3.qkv", 0.02, (q + 2 * kv, hid)).view(np.float16)).to(dev)
    Wo = torch.from_numpy(synth.normal_f16(SEED, "qwen3.o", 0.02, (hid, q)).view(np.float16)).to(dev)
    Wgu = torch.from_numpy(synth.normal_f16(SEED, "qwen3.gu", 0.02, (2 * ffn, hid)).view(np.float16)).to(dev)
    Wd = torch.from_numpy(synth.normal_f16(SEED, "qwen3.down", 0.02, (hid, ffn)).view(np.float16)).to(dev)
    x = torch.from_numpy(synth.normal_f32(SEED, "qwen3.prefill_x", 1.0, (n, hid))).to(dev)
    xo = torch.from_numpy(synth.normal_f16(SEED, "qwen3.prefill_o", 1.0, (n, q)).view(np.float16)).to(dev)
    xf = torch.from_numpy(synth.normal_f32(SEED, "qwen3.prefill_f", 1.0, (n, ffn))).to(dev)
    h = torch.empty((n, hid), dtype=torch.float16, device=dev)
    hf = torch.empty((n, ffn), dtype=torch.float16, device=dev)
    Yqkv = torch.empty((n, q + 2 * kv), dtype=torch.float32, device=dev)
    Yo = torch.empty((n, hid), dtype=torch.float32, device=dev)
    Ygu = torch.empty((n, 2 * ffn), dtype=torch.float32, device=dev)
    Yd = torch.empty((n, hid), dtype=torch.float32, device=dev)
    flops = 2.0 * n * hid * (q + 2 * kv + q + 2 * ffn + ffn)

    def step():
        bm.bm_to_f16(x, h, stream=stream)
        bm.bm_f16_matmul(Wqkv, h, Y=Yqkv, stream=stream)
        bm.bm_f16_matmul(Wo, xo, Y=Yo, stream=stream)
        bm.bm_f16_matmul(Wgu, h, Y=Ygu, stream=stream)
        bm.bm_to_f16(xf, hf, stream=stream)
        bm.bm_f16_matmul(Wd, hf, Y=Yd, stream=stream)

    old = bm.bm_set_pdl(True)
    try:
        ms = graph_time(torch, stream, step, reps=reps)
    finally:
        bm.bm_set_pdl(old)
    return {"tokens": n, "ms_per_step": round(ms, 4), "TFLOP_s": round(flops / ms / 1e9, 1),
            "how": "one layer: Q/K/V and gate/up as one matrix each, O, down, 2 roundings; CUDA graph, PDL on"}


def bench_products(bm, dev, stream, torch):
    """Full-size single products.  One column: a graph of back-to-back products that
    cycle through weight replicas larger than twice the L2 (every launch streams its
    weights from HBM, as in a decode step), programmatic dependent launch on.
    512 columns: one launch after an L2 flush by a read of a 512 MB buffer."""
    out = []
    l2_flush = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    l2_sink = torch.zeros((), dtype=torch.float32, device=dev)

    def flush():
        # a read leaves clean lines, so no write-back lands inside the timed product
        l2_sink.copy_(l2_flush.sum())

    shapes = [("llama3_8b.q", 4096, 4096), ("llama3_8b.gate", 14336, 4096), ("llama3_8b.down", 4096, 14336),
              ("llama3_8b.output", 128256, 4096), ("qwen3_0.6b.logits", 151936, 1024)]
    for name, rows, k in shapes:
        W = torch.from_numpy(synth.normal_f16(SEED, name, 0.01 if "llama" in name else 0.02, (rows, k))
                             .view(np.float16)).to(dev)
        x = torch.from_numpy(synth.normal_f16(SEED, name + ".x", 1.0, (512, k)).view(np.float16)).to(dev)
        nrep = max(2, min(16, -(-2 * 129 * 2 ** 20 // (2 * rows * k))))
        reps = [W] + [W.clone() for _ in range(nrep - 1)]
        y = torch.empty(rows, dtype=torch.float32, device=dev)
        launches = 2 * nrep

        def chain():
            for i in range(launches):
                bm.bm_f16_matvec(reps[i % nrep], x[0], y, stream=stream)

        ms = graph_time(torch, stream, chain) / launches
        gbs = algorithmic_bytes(rows, k) / ms / 1e6
        out.append({"product": name, "rows": rows, "k": k, "ncols": 1, "ms": round(ms, 5), "GB_s": round(gbs, 1),
                    "how": "%d back-to-back launches over %d weight replicas, PDL" % (launches, nrep)})
        few = [(nc, None) for nc in (2, 3, 5, 8, 16, 17, 64)] + [(nc, 8) for nc in (3, 5, 8)] + [(2, 0)]
        for nc, exact_cols in (few if name in ("llama3_8b.q", "llama3_8b.gate") else []):
            # few columns: HBM-bound, timed like the one-column products.  The library's
            # default takes the bit-exact CUDA-core kernel for 2 columns and the tensor
            # cores for more; the (nc, 8) entries time the bit-exact kernel at 3..8 too,
            # the (2, 0) entry the tensor cores at 2.
            Yn = torch.empty((nc, rows), dtype=torch.float32, device=dev)
            xn = x[:nc].contiguous()

            def chain_n():
                for i in range(launches):
                    bm.bm_f16_matmul(reps[i % nrep], xn, Yn, stream=stream)

            old_cols = bm.bm_set_exact_sgemm_cols(exact_cols) if exact_cols is not None else None
            try:
                ms = graph_time(torch, stream, chain_n) / launches
                cur = bm.bm_set_exact_sgemm_cols(0)  # read the setting in force (and put it back)
                bm.bm_set_exact_sgemm_cols(cur)
                exact = nc <= cur
            finally:
                if old_cols is not None:
                    bm.bm_set_exact_sgemm_cols(old_cols)
            out.append({"product": name, "rows": rows, "k": k, "ncols": nc, "ms": round(ms, 5),
                        "GB_s": round(algorithmic_bytes(rows, k, nc) / ms / 1e6, 1),
                        "TFLOP_s": round(2.0 * rows * k * nc / ms / 1e9, 2),
                        "path": "tinyBLAS bit-exact (CUDA cores)" if exact else "tensor cores"})
        Y = torch.empty((512, rows), dtype=torch.float32, device=dev)
        ms = graph_time(torch, stream, lambda: bm.bm_f16_matmul(W, x, Y, stream=stream), reps=5, pre=flush)
        tf = 2.0 * rows * k * 512 / ms / 1e9
        out.append({"product": name, "rows": rows, "k": k, "ncols": 512, "ms": round(ms, 5),
                    "TFLOP_s": round(tf, 1), "GB_s": round(algorithmic_bytes(rows, k, 512) / ms / 1e6, 1)})
        del W, x, y, Y, reps
    out.extend(bench_fallback(bm, dev, stream, torch))
    return out


def bench_fallback(bm, dev, stream, torch):
    """The exact vec_dot kernels off the tinyBLAS path: shapes that fail takes_sgemm
    (13 rows, k % 8 != 0) at 512 columns, and one-column rows of k % 8 != 0 (not
    16-byte aligned, so the lane-per-chain kernel with 2-byte loads), each a graph of
    back-to-back launches cycling through weight replicas larger than twice the L2
    where the weights are large; GB/s of algorithmic bytes against the HBM peak."""
    out = []
    for name, rows, k, nc in (("fallback.13x1536", 13, 1536, 512), ("fallback.4096x33", 4096, 33, 512),
                              ("fallback.12x4097", 12, 4097, 512), ("unaligned.14336x4097", 14336, 4097, 1),
                              ("unaligned.4096x14335", 4096, 14335, 1)):
        W = torch.from_numpy(synth.normal_f16(SEED, name, 0.02, (rows, k)).view(np.float16)).to(dev)
        X = torch.from_numpy(synth.normal_f16(SEED, name + ".x", 1.0, (nc, k)).view(np.float16)).to(dev)
        Y = torch.empty((nc, rows), dtype=torch.float32, device=dev)
        nrep = max(1, min(16, -(-2 * 129 * 2 ** 20 // (2 * rows * k))))
        reps = [W] + [W.clone() for _ in range(nrep - 1)]
        launches = max(8, 2 * nrep)

        def chain():
            for i in range(launches):
                bm.bm_f16_matmul(reps[i % nrep], X, Y, stream=stream)

        ms = graph_time(torch, stream, chain) / launches
        out.append({"product": name, "rows": rows, "k": k, "ncols": nc, "ms": round(ms, 5),
                    "GB_s": round(algorithmic_bytes(rows, k, nc) / ms / 1e6, 1),
                    "TFLOP_s": round(2.0 * rows * k * nc / ms / 1e9, 3),
                    "path": "vec_dot bit-exact (lane per chain)" if nc > 1 else "vec_dot bit-exact (bulk-copied aligned windows)",
                    "how": "%d back-to-back launches over %d weight replicas, PDL" % (launches, nrep)})
        del W, X, Y, reps
    return out


def bench_helpers(bm, dev, stream, torch, launches=8):
    """The standalone pieces around the products, each timed as a CUDA graph of
    `launches` back-to-back calls (PDL on) at a realistic size, as algorithmic bytes /
    time: the RMS norm of a 512-token Llama-3-8B prefill micro-batch (f32 rows in, f32
    and f16 out), the token-embedding lookup of 512 ids from the Llama-3-8B table, and
    the f16 V-accumulator helpers over 64 M elements (larger than L2)."""
    out = []
    gen = torch.Generator(device=dev)
    gen.manual_seed(SEED)

    def timed(name, shape, nbytes, call):
        ms = graph_time(torch, stream, lambda: [call() for _ in range(launches)]) / launches
        out.append({"op": name, "shape": shape, "us": round(ms * 1e3, 2), "GB_s": round(nbytes / ms / 1e6, 1)})

    rows, hid = 512, 4096
    x = torch.randn(rows, hid, device=dev, generator=gen)
    g = torch.rand(hid, device=dev, generator=gen) + 0.5
    y = torch.empty_like(x)
    h = torch.empty(rows, hid, dtype=torch.float16, device=dev)
    timed("bm_rms_norm_mul", "512 x 4096 (f32 and f16 out)", rows * hid * (4 + 4 + 2) + hid * 4,
          lambda: bm.bm_rms_norm_mul(x, g, 1e-5, y, h, stream=stream))
    vocab = 128256
    E = (torch.randn(vocab, hid, device=dev, generator=gen) * 0.01).to(torch.float16)
    ids = torch.randint(0, vocab, (rows,), device=dev, dtype=torch.int32, generator=gen)
    emb = torch.empty(rows, hid, dtype=torch.float32, device=dev)
    timed("bm_f16_get_rows", "512 ids of 128256 x 4096", rows * hid * (2 + 4) + rows * 4,
          lambda: bm.bm_f16_get_rows(E, ids, emb, stream=stream))
    n = 64 << 20
    acc = (torch.randn(n, device=dev, generator=gen) * 0.1).to(torch.float16)
    v = (torch.randn(n, device=dev, generator=gen) * 0.1).to(torch.float16)
    timed("bm_f16_mad", "64 M elements", 6 * n, lambda: bm.bm_f16_mad(acc, v, 0.999, stream=stream))
    timed("bm_f16_scale", "64 M elements", 4 * n, lambda: bm.bm_f16_scale(acc, 1.0001, stream=stream))
    del x, y, h, E, ids, emb, acc, v
    return out


# ----------------------------------------------------------------------------- CPU oracle


def oracle_sample_runner(model=HEADLINE):
    """A bounded sample of the decode step on the CPU oracle: one layer's four calls (every
    layer has the same shapes) and 1/L of the head's rows, with the step's own weights and
    activations.  Returns (run_one_sample, bytes_per_sample, threads, description)."""
    import oracle

    spec = MODELS[model]
    L = spec["layers"]
    plan = step_plan(model)
    layer0 = plan[:4]
    head = plan[-1]
    hk, hrows = head[2], -(-head[1][0][2] // L)
    weights = {}
    for _, mats, k, _ in layer0:
        for _, wn, rows in mats:
            weights[wn] = synth.normal_f16(SEED, wn, spec["sigma"], (rows, k))
    hw = synth.normal_f16(SEED, head[1][0][1], spec["sigma"], (hrows, hk))  # the head's first rows (counter-based)
    acts = {a: synth.normal_f32(SEED, act_name(model, a), A_SIGMA, k) for _, _, k, a in layer0 + [head]}
    nbytes = step_bytes(layer0, True) + 2 * hrows * hk + 4 * hrows + 4 * hk

    def run():
        for kind, mats, k, a in layer0:
            h = oracle.to_f16(acts[a])
            if kind == "multi":
                oracle.matvec_multi([weights[wn] for _, wn, _ in mats], h)
            else:
                oracle.matvec(weights[mats[0][1]], h)
        oracle.matvec(hw, oracle.to_f16(acts[head[3]]))

    desc = ("one layer's 4 calls (Q/K/V, O, gate/up, down; %.0f MB of f16 weights) and %d of the %d head rows "
            "(1/%d) of the %s decode step, activations rounded by the oracle" %
            (weight_bytes(layer0) / 1e6, hrows, head[1][0][2], L, model))
    return run, nbytes, oracle.threads(), desc


def host_cpu():
    """The host's architecture and CPU model, as the kernel reports them."""
    import platform
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware") and not model:
                    model = line.split(":", 1)[1].strip()
    except OSError:
        pass
    return {"machine": platform.machine(), "cpu": model, "logical_cpus": os.cpu_count()}


def cpu_baseline(budget_s=10.0, budget_1core_s=4.0):
    import oracle
    run, nbytes, cores, desc = oracle_sample_runner()

    def timed(budget):
        run()
        n = 0
        t0 = time.perf_counter()
        while True:
            run()
            n += 1
            if time.perf_counter() - t0 >= budget:
                break
        return n, time.perf_counter() - t0

    n, dt = timed(budget_s)
    oracle.set_threads(1)
    try:
        n1, dt1 = timed(budget_1core_s)
    finally:
        oracle.set_threads(cores)
    # the largest products on all cores: a deterministic subset of rows, the time scaled
    # per row to the whole matrix (extrapolated, and said so)
    products = []
    for name, rows, k, nc, sub in (("llama3_8b.output", 128256, 4096, 512, 32), ("llama3_8b.gate", 14336, 4096, 1, 2048)):
        W = synth.normal_f16(SEED, "cpu." + name, 0.01, (sub, k))
        X = oracle.to_f16(synth.normal_f32(SEED, "cpu." + name + ".x", 1.0, (nc, k)))
        t0 = time.perf_counter()
        if nc == 1:
            oracle.matvec(W, X[0])
        else:
            oracle.matmul(W, X)
        full_s = (time.perf_counter() - t0) * rows / sub
        entry = {"product": name, "rows": rows, "k": k, "ncols": nc, "rows_timed": sub,
                 "seconds_extrapolated": round(full_s, 3)}
        if nc == 1:
            entry["GB_s"] = round(algorithmic_bytes(rows, k) / full_s / 1e9, 2)
        else:
            entry["TFLOP_s"] = round(2.0 * rows * k * nc / full_s / 1e12, 5)
        products.append(entry)
    return {"value": round(nbytes * n / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d repetitions in %.1f s on the host of %s" % (n, dt, desc),
            "value_1core": round(nbytes * n1 / dt1 / 1e9, 4),
            "sample_1core": "%d repetitions in %.1f s on one core" % (n1, dt1), "host": host_cpu(),
            "products": products}


def step_config(model=HEADLINE, layers=None):
    """The workload both arms measure (a description of the data, not of how it runs)."""
    spec = MODELS[model]
    plan = step_plan(model, layers)
    return {"workload": "%s_decode_step" % model, "layers": spec["layers"] if layers is None else layers,
            "hidden": spec["hidden"], "q_rows": spec["q"], "kv_rows": spec["kv"], "ffn": spec["ffn"],
            "vocab": spec["vocab"], "ncols": 1, "calls_per_step": len(plan), "seed": SEED,
            "weight_sigma": spec["sigma"], "activation_sigma": A_SIGMA, "weight_bytes": weight_bytes(plan),
            "algorithmic_bytes_per_step": step_bytes(plan, True)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    run, nbytes, cores, desc = oracle_sample_runner()
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    value = nbytes / (ms / 1e3) / 1e9
    cfg = step_config()
    cfg.update({"runs_on": "host CPU cores (OpenMP over output rows)", "l2": None,
                "step_sample": "each step is a bounded sample: " + desc})
    line = {
        "impl": "reference", "metric": "decode F16 GEMV HBM GB/s (Llama-3-8B-shaped decode step)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 weights and activations, f32 accumulate (vec_dot bits)", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "%d steps after %d warm-up, each %s" % (args.steps, args.warmup, desc)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- profile modes


def run_single(spec: str, reps: int):
    """One product ROWSxKxNCOLS, `reps` times (for profilers; prints nothing timed)."""
    import torch

    import __graft_entry__
    import f16_weight_gemv_gb300 as bm

    __graft_entry__.build()
    rows, k, ncols = (int(v) for v in spec.lower().split("x"))
    dev = torch.device("cuda", 0)
    W = torch.from_numpy(synth.normal_f16(SEED, "single.w", 0.02, (rows, k)).view(np.float16)).to(dev)
    X = torch.from_numpy(synth.normal_f16(SEED, "single.x", A_SIGMA, (ncols, k)).view(np.float16)).to(dev)
    Y = torch.empty((ncols, rows), dtype=torch.float32, device=dev)
    for _ in range(reps):
        if ncols == 1:
            bm.bm_f16_matvec(W, X[0], Y[0])
        else:
            bm.bm_f16_matmul(W, X, Y)
    torch.cuda.synchronize()
    print(json.dumps({"single": spec, "reps": reps, "status": bm.bm_device_status()}))
    return 0


def run_decode(spec: str, reps: int):
    """MODEL:LAYERS -- that decode step with LAYERS layers (and the head), eagerly, `reps`
    times with programmatic dependent launch on (for profilers; prints nothing timed).
    Each product's shape is the full step's, so its per-launch counters are too."""
    import torch

    import __graft_entry__
    import f16_weight_gemv_gb300 as bm

    __graft_entry__.build()
    model, layers = spec.split(":")
    dev = torch.device("cuda", 0)
    bm.bm_set_pdl(True)
    step = DecodeStep(bm, torch, dev, model, int(layers))
    s = torch.cuda.current_stream()
    for _ in range(reps):
        step.run(s)
    torch.cuda.synchronize()
    print(json.dumps({"decode": spec, "launches_per_step": len(step.plan), "reps": reps,
                      "keys": [call_key(m, k) for _, m, k, _ in step.plan], "status": bm.bm_device_status()}))
    return 0


def run_helper(name: str, reps: int):
    """One of the bench's helpers (bench_helpers) at its size, `reps` times (for
    profilers; prints nothing timed): mad, scale, norm or get_rows."""
    import torch

    import __graft_entry__
    import f16_weight_gemv_gb300 as bm

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(SEED)
    if name in ("mad", "scale"):
        n = 64 << 20
        acc = (torch.randn(n, device=dev, generator=gen) * 0.1).to(torch.float16)
        v = (torch.randn(n, device=dev, generator=gen) * 0.1).to(torch.float16)
        call = (lambda: bm.bm_f16_mad(acc, v, 0.999)) if name == "mad" else (lambda: bm.bm_f16_scale(acc, 1.0001))
    elif name == "norm":
        x = torch.randn(512, 4096, device=dev, generator=gen)
        g = torch.rand(4096, device=dev, generator=gen) + 0.5
        y = torch.empty_like(x)
        h = torch.empty(512, 4096, dtype=torch.float16, device=dev)
        call = lambda: bm.bm_rms_norm_mul(x, g, 1e-5, y, h)  # noqa: E731
    elif name == "get_rows":
        E = (torch.randn(128256, 4096, device=dev, generator=gen) * 0.01).to(torch.float16)
        ids = torch.randint(0, 128256, (512,), device=dev, dtype=torch.int32, generator=gen)
        out = torch.empty(512, 4096, dtype=torch.float32, device=dev)
        call = lambda: bm.bm_f16_get_rows(E, ids, out)  # noqa: E731
    else:
        raise SystemExit("unknown helper " + name)
    for _ in range(reps):
        call()
    torch.cuda.synchronize()
    print(json.dumps({"helper": name, "reps": reps, "status": bm.bm_device_status()}))
    return 0


def run_prefill(reps: int):
    """The Llama-3-8B-shaped prefill layer (PrefillLayer, bm_f16_matmul_multi variant),
    eagerly, `reps` times with programmatic dependent launch on (for profilers; prints
    nothing timed)."""
    import torch

    import __graft_entry__
    import f16_weight_gemv_gb300 as bm

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    layer = PrefillLayer(bm, torch, dev)
    bm.bm_set_pdl(True)
    s = torch.cuda.current_stream()
    for _ in range(reps):
        layer.run(s, "multi")
    torch.cuda.synchronize()
    print(json.dumps({"prefill": "llama3_8b layer, 512 tokens", "reps": reps, "status": bm.bm_device_status()}))
    return 0


# ----------------------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--single", default=None, help="profile mode: run one product ROWSxKxNCOLS --reps times")
    ap.add_argument("--decode", default=None, help="profile mode: run the decode step MODEL:LAYERS --reps times")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--prefill", action="store_true", help="profile mode: run the Llama-3-8B prefill layer --reps times")
    ap.add_argument("--helper", default=None, choices=["mad", "scale", "norm", "get_rows"],
                    help="profile mode: run one of the helpers --reps times")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-layers", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--no-products", action="store_true", help="the headline objects only")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.single:
        return run_single(args.single, args.reps)
    if args.decode:
        return run_decode(args.decode, args.reps)
    if args.prefill:
        return run_prefill(args.reps)
    if args.helper:
        return run_helper(args.helper, args.reps)

    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    import __graft_entry__
    if rank == 0 or not os.path.exists(os.path.join(ROOT, "f16_weight_gemv_gb300", "libbm.so")):
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()

    r = run_gpu(args, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return 0

    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    hbm_src = "measured (MEASURED_PEAKS.json hbm_gbs)" if "hbm_gbs" in peaks else "fallback 6.8 TB/s"
    tc_peak = float(peaks.get("bf16_tflops", 1900.0))
    tc_src = ("measured (MEASURED_PEAKS.json bf16_tflops, burst: the layer is timed alone); f16 and bf16 run at "
              "the same dense rate" if "bf16_tflops" in peaks else "fallback 1.9 PFLOP/s")
    value = r["tot_bytes"] * world / (r["ms"] / 1e3) / 1e9
    achieved = r["tot_bytes"] / (r["ms"] / 1e3) / 1e9
    layers = args.decode_layers
    cfg = step_config(HEADLINE, layers)
    cfg.update({"l2": "inputs larger than L2: %.1f GB of weights per step, read once per step" %
                      (r["weight_bytes"] / 1e9),
                "parallelism": "replicas" if world > 1 else "single GPU", "graph": "CUDA graph of the step",
                "pdl": not args.no_pdl})
    gb = lambda ms: round(r["tot_bytes"] / (ms / 1e3) / 1e9, 2)  # noqa: E731
    line = {
        "metric": "decode F16 GEMV HBM GB/s (Llama-3-8B-shaped decode step)",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(r["ms"], 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 weights and activations, f32 accumulate (vec_dot bits)", "data": "synthetic",
        "config": cfg,
        "pct_of_hbm_peak": round(100.0 * value / world / hbm_peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": ncu_traffic_per_launch(r["plan"]),
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                     "algorithmic_bytes_per_launch": int(r["tot_bytes"] / r["launches_per_step"]),
                     "kernel": "k_gemv_stream (rounding + one-column GEMV)", "peak_source": hbm_src,
                     "launches_per_step": r["launches_per_step"],
                     "how": "the step's only kernel: algorithmic bytes of its launches / CUDA-event time of the "
                            "step graph's replays on the launch stream"},
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": r["clocks"],
        "e2e": {"value": gb(r["ms_e2e"]), "unit": "GB/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "ms_per_step": round(r["ms_e2e"], 5),
                "how": "every step: the step's f32 activations copied from pinned host memory, the 129 calls "
                       "recorded once by the binding's prepare() made one C call each, the logits copied back to "
                       "pinned host memory and waited for on the host; wall clock",
                "graph_value": gb(r["ms_e2e_graph"]),
                "graph_how": "the same with the recorded calls captured once as a CUDA graph (Prepared.graph())",
                "eager_value": gb(r["ms_e2e_eager"]),
                "eager_how": "the same with every call made through the wrappers (argument checks each time)"},
        "one_launch": {"ms_per_step": round(r["ms_one"], 5), "GB_s": gb(r["ms_one"]),
                       "how": "the same 129 calls recorded once (bm_step_create) and run as one cooperative launch "
                              "(bm_step_run), each call waiting on the device for every earlier call; CUDA events"},
        "device": torch.cuda.get_device_name(),
    }
    if "prefill" in r:
        pf = r["prefill"]
        line["prefill"] = {
            "metric": "prefill GEMM TFLOP/s (% of dense FP16 peak)", "value": pf["TFLOP_s"], "unit": "TFLOP/s",
            "pct_of_peak": round(100.0 * pf["TFLOP_s"] / tc_peak, 1),
            "roofline": {"bound": "tensor", "achieved": pf["TFLOP_s"], "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": round(pf["TFLOP_s"] / tc_peak, 4), "traffic": prefill_traffic_per_launch(),
                         "traffic_unit": "bytes per k_gemm_tc launch of the layer (ncu dram__bytes_read.sum + "
                                         "dram__bytes_write.sum, mean of its 4 launches)",
                         "algorithmic_bytes_per_launch": int(round(sum(
                             2 * r * k + 2 * k * 512 + 4 * r * 512 for r, k in
                             ((6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336))) / 4)),
                         "kernel": "k_gemm_tc (tcgen05 + TMA + TMEM)", "peak_source": tc_src,
                         "how": "the layer's algorithmic flops / CUDA-event time of the whole layer graph, which also "
                                "holds the two rounding kernels and the split-k reductions: a lower bound on the "
                                "tensor-core kernel's own rate"},
            **pf}
        for p in pf["products"]:
            p["pct_of_peak"] = round(100.0 * p["TFLOP_s"] / tc_peak, 1)
    for key in ("smollm2_135m_decode_step", "qwen3_0.6b_decode_step"):
        if key in r:
            r[key]["pct_hbm"] = round(100.0 * r[key]["GB_s"] / hbm_peak, 1)
            line[key] = r[key]
    if "qwen3_0.6b_prefill_layer" in r:
        pq = r["qwen3_0.6b_prefill_layer"]
        pq["pct_bf16_dense_peak"] = round(100.0 * pq["TFLOP_s"] / tc_peak, 1)
        line["qwen3_0.6b_prefill_layer"] = pq
    if "helpers" in r:
        for p in r["helpers"]:
            p["pct_hbm"] = round(100.0 * p["GB_s"] / hbm_peak, 1)
        line["helpers"] = r["helpers"]
    if "products" in r:
        line["products"] = r["products"]
        for p in r["products"]:
            if p["ncols"] <= 64 or "path" in p and "vec_dot" in p["path"]:
                p["pct_hbm"] = round(100.0 * p["GB_s"] / hbm_peak, 1)
            else:
                p["pct_bf16_dense_peak"] = round(100.0 * p["TFLOP_s"] / tc_peak, 1)
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
