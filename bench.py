#!/usr/bin/env python3
"""Benchmark of the F16-weight products on one GB300 (or N replicas).

Default workload: a SmolLM2-135M-shaped decode step -- 30 layers of
[fused Q/K/V product (576+192+192 rows x 576), O (576 x 576), fused gate/up
(2 x 1536 x 576), down (576 x 1536)] then the tied logits (49152 x 576): one
column, 121 products over 269 MB of f16 weights (more than the 129 MB L2),
seeded synthetic weights N(0, 0.02) and f32 activations N(0, 1).  Each product
is one bm_f16_matvec_act call: the f32 activation is rounded to f16 and
multiplied in the same launch.  The step is captured once as a CUDA graph
(programmatic dependent launch on) and replayed; `value` is algorithmic bytes
per step / time per step.

Extra objects in the same JSON line:
  roofline     -- the step's kernel (k_gemv_stream) against the measured HBM peak
  unfused      -- the same step as bm_to_f16 + bm_f16_matvec[_multi]/bm_f16_logits
                  (242 launches)
  norm_front_end -- the step with the RMS norm ahead of Q/K/V, gate/up and the
                  logits fused into those products (bm_f16_matvec_norm)
  products     -- single products of the Llama-3-8B / Qwen3-0.6B shapes:
                  decode GB/s and 512-column tensor-core TFLOP/s
  llama3_8b_decode_step / llama3_8b_prefill_layer -- a whole Llama-3-8B-shaped
                  decode step (129 products), and one layer's 7 products for a
                  512-token prefill micro-batch (with and without PDL)
  e2e          -- the same step through the Python binding without a graph (the
                  step's calls recorded once by prepare(), replayed each step; and
                  made through the wrappers each time), with the step's activations
                  copied from pinned host memory and the logits copied back every step
  cpu_baseline -- the CPU oracle on this host, full decode steps

`--impl reference` times the CPU oracle (the only reference that exists for
this method) on the same workload and prints the same JSON line.
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

HIDDEN, FFN, VOCAB, LAYERS = 576, 1536, 49152, 30
Q_ROWS, KV_ROWS = 9 * 64, 3 * 64
SEED = 0
W_SIGMA, A_SIGMA = 0.02, 1.0


# DRAM traffic per launch of the step's kernel, from the ncu launch list of one
# timed step (profiles/decode_step_smollm2_launches.md), valid only for the kernel
# source it was measured on (sha256 prefix of k_gemv_stream.cu).
NCU_TRAFFIC = {"kernel": "k_gemv_stream", "source": "f16_weight_gemv_gb300/csrc/k_gemv_stream.cu",
               "sha256_16": "78fefbba59017a3a", "bytes_per_launch": 2294604}


def ncu_traffic():
    import hashlib
    try:
        with open(os.path.join(ROOT, NCU_TRAFFIC["source"]), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None
    return NCU_TRAFFIC["bytes_per_launch"] if sha == NCU_TRAFFIC["sha256_16"] else None


def algorithmic_bytes(rows, k, ncols=1):
    return 2 * rows * k + 2 * k * ncols + 4 * rows * ncols


def step_plan():
    """The decode step as an ordered list of calls: ('round', n, act_id) or
    ('multi'|'mv'|'logits', [(name, rows)], k, act_id)."""
    plan = []
    a = 0
    for L in range(LAYERS):
        plan.append(("round", HIDDEN, a))
        plan.append(("multi", [("l%d.q" % L, Q_ROWS), ("l%d.k" % L, KV_ROWS), ("l%d.v" % L, KV_ROWS)], HIDDEN, a))
        a += 1
        plan.append(("round", HIDDEN, a))
        plan.append(("mv", [("l%d.o" % L, HIDDEN)], HIDDEN, a))
        a += 1
        plan.append(("round", HIDDEN, a))
        plan.append(("multi", [("l%d.gate" % L, FFN), ("l%d.up" % L, FFN)], HIDDEN, a))
        a += 1
        plan.append(("round", FFN, a))
        plan.append(("mv", [("l%d.down" % L, HIDDEN)], FFN, a))
        a += 1
    plan.append(("round", HIDDEN, a))
    plan.append(("logits", [("token_embd", VOCAB)], HIDDEN, a))
    return plan


def step_bytes(plan, fused=True):
    """Algorithmic bytes of one step.  Fused: each product call reads its f32
    activation (4k) and rounds it in the kernel; unfused: a rounding call (6 bytes
    per element) then the product reads the f16 activation (2k).  Weights 2*rows*k
    and outputs 4*rows either way; a fused multi-matrix call reads its activation once."""
    tot = 0
    for op in plan:
        if op[0] == "round":
            tot += 0 if fused else 6 * op[1]
        else:
            k = op[2]
            tot += sum(2 * r * k + 4 * r for _, r in op[1]) + (4 * k if fused else 2 * k)
    return tot


def act_sizes(plan):
    sizes = {}
    for op in plan:
        if op[0] == "round":
            sizes[op[2]] = op[1]
    return sizes


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
                                          "-i", str(self.index), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

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
        inside = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15] or rows[-3:]
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


# ----------------------------------------------------------------------------- GPU arm


def run_gpu(args, rank, world, local_rank):
    import torch

    import f16_weight_gemv_gb300 as bm

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    bm.lib()
    plan = step_plan()
    tot_bytes, unfused_bytes = step_bytes(plan, True), step_bytes(plan, False)

    # ---- weights and activations (seeded, generated on the host once, then resident)
    weights = {}
    for op in plan:
        if op[0] == "round":
            continue
        for name, rows in op[1]:
            w = synth.normal_f16(SEED, "smollm2." + name, W_SIGMA, (rows, op[2]))
            weights[name] = torch.from_numpy(w.view(np.float16)).to(dev)
    sizes = act_sizes(plan)
    offs, o = {}, 0
    for a in sorted(sizes):
        offs[a] = o
        o += (sizes[a] + 7) // 8 * 8  # 32-byte aligned slices
    act_host = np.zeros(o, dtype=np.float32)
    for a in sorted(sizes):
        act_host[offs[a]:offs[a] + sizes[a]] = synth.normal_f32(SEED, "smollm2.act%d" % a, A_SIGMA, sizes[a])
    act_f32 = torch.from_numpy(act_host).to(dev)
    act_f16 = torch.empty(o, dtype=torch.float16, device=dev)
    outs = {}
    for op in plan:
        if op[0] != "round":
            for name, rows in op[1]:
                outs[name] = torch.empty(rows, dtype=torch.float32, device=dev)

    stream = torch.cuda.Stream(device=dev)
    # The weights are constants: programmatic dependent launch lets each product start
    # copying its weights while the kernel ahead of it is still running.
    bm.bm_set_pdl(not args.no_pdl)

    norm_w = {k: torch.from_numpy((1.0 + synth.normal_f32(SEED, "smollm2.norm%d" % k, 0.2, k))
                                  .astype(np.float32)).to(dev) for k in (HIDDEN,)}

    def run_step(s, fused=True, norm=False):
        for op in plan:
            if op[0] == "round":
                if not fused:
                    a = op[2]
                    bm.bm_to_f16(act_f32[offs[a]:offs[a] + op[1]], act_f16[offs[a]:offs[a] + op[1]], stream=s)
                continue
            kind, mats, k, a = op
            if norm and kind in ("multi", "logits"):
                # the norm ahead of Q/K/V, of gate/up and of the logits, fused into the product
                bm.bm_f16_matvec_norm([weights[n] for n, _ in mats], act_f32[offs[a]:offs[a] + k], norm_w[k], 1e-5,
                                      [outs[n] for n, _ in mats], stream=s)
                continue
            if fused:
                bm.bm_f16_matvec_act([weights[n] for n, _ in mats], act_f32[offs[a]:offs[a] + k],
                                     [outs[n] for n, _ in mats], stream=s)
                continue
            x = act_f16[offs[a]:offs[a] + k]
            if kind == "multi":
                bm.bm_f16_matvec_multi([weights[n] for n, _ in mats], x, [outs[n] for n, _ in mats], stream=s)
            elif kind == "mv":
                bm.bm_f16_matvec(weights[mats[0][0]], x, outs[mats[0][0]], stream=s)
            else:
                bm.bm_f16_logits(weights[mats[0][0]], x.view(1, -1), outs[mats[0][0]].view(1, -1), stream=s)

    launches_per_step = sum(1 for op in plan if op[0] != "round")

    def capture(fused, norm=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            run_step(stream, fused, norm)  # warm (attribute setup happens outside capture)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            run_step(stream, fused, norm)
        torch.cuda.synchronize()
        return g

    g_step = capture(True)
    g_unfused = capture(False)
    g_norm = capture(True, True)

    def timed(g, steps, warmup):
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
        return e0.elapsed_time(e1) / steps  # ms per step

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else
                          int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank]))
    clocks.start()
    time.sleep(0.3)
    t_begin = time.time()
    ms = timed(g_step, args.steps, args.warmup)
    t_end = time.time()
    ms_unfused = timed(g_unfused, max(args.steps, 20), args.warmup)
    ms_norm = timed(g_norm, max(args.steps, 20), args.warmup)
    clk = clocks.summary(t_begin, t_end)
    clocks.stop()

    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())

    # ---- end to end through the binding: pinned H2D of the step's activations, eager
    # calls, D2H of the logits, every step
    act_pinned = torch.from_numpy(act_host).pin_memory()
    logits_host = torch.empty(VOCAB, dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))

    # the step's 121 calls recorded once through the binding's prepare(): each replay is
    # one C call per product (the same entry points, pointers and stream)
    prepared = bm.prepare(lambda: run_step(stream))

    def e2e_step(calls):
        with torch.cuda.stream(stream):
            act_f32.copy_(act_pinned, non_blocking=True)
            calls()
            logits_host.copy_(outs["token_embd"], non_blocking=True)

    def e2e_time(calls):
        for _ in range(2):
            e2e_step(calls)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step(calls)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / e2e_steps

    prepared_graph = prepared.graph(stream)
    ms_e2e = e2e_time(prepared_graph)
    ms_e2e_replay = e2e_time(prepared)
    ms_e2e_eager = e2e_time(lambda: run_step(stream))

    result = {
        "ms": ms, "ms_unfused": ms_unfused, "ms_norm": ms_norm, "ms_e2e": ms_e2e, "ms_e2e_replay": ms_e2e_replay,
        "ms_e2e_eager": ms_e2e_eager, "tot_bytes": tot_bytes,
        "unfused_bytes": unfused_bytes, "launches_per_step": launches_per_step, "clocks": clk,
        "h2d": int(act_host.nbytes), "d2h": int(VOCAB * 4),
    }
    if rank == 0 and not args.no_products:
        result["products"] = bench_products(bm, dev, stream, torch)
        result["llama3_8b_decode_step"] = bench_llama_decode(bm, dev, stream, torch)
        result["llama3_8b_prefill_layer"] = bench_llama_prefill(bm, dev, stream, torch)
        result["qwen3_0.6b_decode_step"] = bench_qwen3_decode(bm, dev, stream, torch)
        result["qwen3_0.6b_prefill_layer"] = bench_qwen3_prefill(bm, dev, stream, torch)
        result["helpers"] = bench_helpers(bm, dev, stream, torch)
    return result


def graph_time(torch, stream, fn, reps=3, pre=None):
    """Capture fn() once as a CUDA graph; median ms of `reps` replays (pre() runs
    before each replay, outside the timed events)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
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
    return out


def bench_llama_decode(bm, dev, stream, torch, steps=10):
    """A Llama-3-8B-shaped decode step: 32 layers of [fused Q/K/V (4096+1024+1024 x
    4096), O (4096 x 4096), fused gate/up (2 x 14336 x 4096), down (4096 x 14336)]
    then the output product (128256 x 4096): 129 bm_f16_matvec_act calls over 15 GB
    of f16 weights N(0, 0.01).  One layer's weights are drawn and copied to all 32
    layers (distinct memory: every product still streams from HBM)."""
    hid, ffn, kv, vocab, layers = 4096, 14336, 1024, 128256, 32
    base = {n: torch.from_numpy(synth.normal_f16(SEED, "llama3_8b." + n, 0.01, (r, c)).view(np.float16)).to(dev)
            for n, r, c in [("q", hid, hid), ("k", kv, hid), ("v", kv, hid), ("o", hid, hid), ("gate", ffn, hid),
                            ("up", ffn, hid), ("down", hid, ffn)]}
    lw = [{n: (t if L == 0 else t.clone()) for n, t in base.items()} for L in range(layers)]
    out_w = torch.from_numpy(synth.normal_f16(SEED, "llama3_8b.output", 0.01, (vocab, hid)).view(np.float16)).to(dev)
    xa = torch.from_numpy(synth.normal_f32(SEED, "llama3_8b.act", 1.0, hid)).to(dev)
    xf = torch.from_numpy(synth.normal_f32(SEED, "llama3_8b.act_ffn", 1.0, ffn)).to(dev)
    ys = {n: torch.empty(t.shape[0], dtype=torch.float32, device=dev) for n, t in base.items()}
    logits = torch.empty(vocab, dtype=torch.float32, device=dev)
    nbytes = 0
    for n, t in base.items():
        nbytes += layers * (2 * t.numel() + 4 * t.shape[0])
    nbytes += layers * 4 * (hid + hid + hid + ffn) + 2 * vocab * hid + 4 * vocab + 4 * hid

    def step():
        for L in range(layers):
            w = lw[L]
            bm.bm_f16_matvec_act([w["q"], w["k"], w["v"]], xa, [ys["q"], ys["k"], ys["v"]], stream=stream)
            bm.bm_f16_matvec_act([w["o"]], xa, [ys["o"]], stream=stream)
            bm.bm_f16_matvec_act([w["gate"], w["up"]], xa, [ys["gate"], ys["up"]], stream=stream)
            bm.bm_f16_matvec_act([w["down"]], xf, [ys["down"]], stream=stream)
        bm.bm_f16_matvec_act([out_w], xa, [logits], stream=stream)

    norms = [torch.from_numpy((1.0 + synth.normal_f32(SEED, "llama3_8b.norm%d" % i, 0.2, hid)).astype(np.float32))
             .to(dev) for i in range(2 * layers + 1)]

    def step_norm():
        # the same step with the RMS norm ahead of Q/K/V, gate/up and the output product
        # fused into those launches (each reads its norm weight, 4 * 4096 bytes, too)
        for L in range(layers):
            w = lw[L]
            bm.bm_f16_matvec_norm([w["q"], w["k"], w["v"]], xa, norms[2 * L], 1e-5, [ys["q"], ys["k"], ys["v"]],
                                  stream=stream)
            bm.bm_f16_matvec_act([w["o"]], xa, [ys["o"]], stream=stream)
            bm.bm_f16_matvec_norm([w["gate"], w["up"]], xa, norms[2 * L + 1], 1e-5, [ys["gate"], ys["up"]],
                                  stream=stream)
            bm.bm_f16_matvec_act([w["down"]], xf, [ys["down"]], stream=stream)
        bm.bm_f16_matvec_norm([out_w], xa, norms[-1], 1e-5, [logits], stream=stream)

    ms = graph_time(torch, stream, step, reps=steps)
    ms_norm = graph_time(torch, stream, step_norm, reps=steps)
    res = {"ms_per_step": round(ms, 4), "GB_s": round(nbytes / ms / 1e6, 1), "weight_GB": round(
        (sum(t.numel() for t in base.values()) * layers + out_w.numel()) * 2 / 1e9, 3), "launches": 4 * layers + 1,
        "with_norm_front_end": {"ms_per_step": round(ms_norm, 4),
                                "GB_s": round((nbytes + 4 * hid * (2 * layers + 1)) / ms_norm / 1e6, 1),
                                "how": "bm_f16_matvec_norm for Q/K/V, gate/up and the output product"}}
    del lw, out_w, base, norms
    return res


def bench_qwen3_decode(bm, dev, stream, torch, steps=10):
    """A Qwen3-0.6B-shaped decode step: 28 layers of [fused Q/K/V (2048+1024+1024 x 1024),
    O (1024 x 2048), fused gate/up (2 x 3072 x 1024), down (1024 x 3072)] then the tied
    logits (151936 x 1024): 113 bm_f16_matvec_act calls over 1.19 GB of f16 weights
    N(0, 0.02), one layer drawn and copied to 28 distinct buffers."""
    hid, q, kv, ffn, vocab, layers = 1024, 2048, 1024, 3072, 151936, 28
    base = {n: torch.from_numpy(synth.normal_f16(SEED, "qwen3." + n, 0.02, (r, c)).view(np.float16)).to(dev)
            for n, r, c in [("q", q, hid), ("k", kv, hid), ("v", kv, hid), ("o", hid, q), ("gate", ffn, hid),
                            ("up", ffn, hid), ("down", hid, ffn)]}
    lw = [{n: (t if L == 0 else t.clone()) for n, t in base.items()} for L in range(layers)]
    emb = torch.from_numpy(synth.normal_f16(SEED, "qwen3.embd", 0.02, (vocab, hid)).view(np.float16)).to(dev)
    xa = torch.from_numpy(synth.normal_f32(SEED, "qwen3.act", 1.0, hid)).to(dev)
    xo = torch.from_numpy(synth.normal_f32(SEED, "qwen3.act_o", 1.0, q)).to(dev)
    xf = torch.from_numpy(synth.normal_f32(SEED, "qwen3.act_ffn", 1.0, ffn)).to(dev)
    ys = {n: torch.empty(t.shape[0], dtype=torch.float32, device=dev) for n, t in base.items()}
    logits = torch.empty(vocab, dtype=torch.float32, device=dev)
    nbytes = 0
    for n, t in base.items():
        nbytes += layers * (2 * t.numel() + 4 * t.shape[0])
    nbytes += layers * 4 * (hid + q + hid + ffn) + 2 * vocab * hid + 4 * vocab + 4 * hid

    def step():
        for L in range(layers):
            w = lw[L]
            bm.bm_f16_matvec_act([w["q"], w["k"], w["v"]], xa, [ys["q"], ys["k"], ys["v"]], stream=stream)
            bm.bm_f16_matvec_act([w["o"]], xo, [ys["o"]], stream=stream)
            bm.bm_f16_matvec_act([w["gate"], w["up"]], xa, [ys["gate"], ys["up"]], stream=stream)
            bm.bm_f16_matvec_act([w["down"]], xf, [ys["down"]], stream=stream)
        bm.bm_f16_matvec_act([emb], xa, [logits], stream=stream)

    ms = graph_time(torch, stream, step, reps=steps)
    res = {"ms_per_step": round(ms, 4), "GB_s": round(nbytes / ms / 1e6, 1), "weight_GB": round(
        (sum(t.numel() for t in base.values()) * layers + emb.numel()) * 2 / 1e9, 3), "launches": 4 * layers + 1}
    del lw, emb, base
    return res


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


def bench_llama_prefill(bm, dev, stream, torch, reps=10):
    """A Llama-3-8B-shaped prefill micro-batch of 512 tokens through one layer's products:
    the rounding of the normed activations, Q/K/V/O (4096, 1024, 1024, 4096 rows x 4096),
    gate and up (14336 x 4096), the rounding of the FFN activation and down (4096 x 14336):
    7 tensor-core products and 2 rounding kernels per step (plus a reduction after each
    product that splits k), one CUDA graph, with and without programmatic dependent launch.
    The layer's 436 MB of weights exceed L2, so replays stream them from HBM."""
    hid, ffn, kv, n = 4096, 14336, 1024, 512
    shapes = [("q", hid, hid), ("k", kv, hid), ("v", kv, hid), ("o", hid, hid), ("gate", ffn, hid),
              ("up", ffn, hid), ("down", hid, ffn)]
    W = {nm: torch.from_numpy(synth.normal_f16(SEED, "llama3_8b." + nm, 0.01, (r, c)).view(np.float16)).to(dev)
         for nm, r, c in shapes}
    x = torch.from_numpy(synth.normal_f32(SEED, "llama3_8b.prefill_x", 1.0, (n, hid))).to(dev)
    h = torch.empty((n, hid), dtype=torch.float16, device=dev)
    Y = {nm: torch.empty((n, r), dtype=torch.float32, device=dev) for nm, r, _ in shapes}
    hd = torch.empty((n, ffn), dtype=torch.float16, device=dev)
    flops = 2.0 * n * sum(r * c for _, r, c in shapes)

    def step():
        bm.bm_to_f16(x, h, stream=stream)
        for nm in ("q", "k", "v", "o", "gate", "up"):
            bm.bm_f16_matmul(W[nm], h, Y=Y[nm], stream=stream)
        bm.bm_to_f16(Y["gate"], hd, stream=stream)
        bm.bm_f16_matmul(W["down"], hd, Y=Y["down"], stream=stream)

    # The same layer with Q/K/V and gate/up stored as one matrix each ([6144][4096] and
    # [28672][4096]): two products instead of five.  Every element is still its own row's
    # product (the path follows the concatenated shape, which takes_sgemm the same way),
    # and a caller reads Q, K, V (or gate, up) as row ranges of each output column.
    Wqkv = torch.cat([W["q"], W["k"], W["v"]], 0)
    Wgu = torch.cat([W["gate"], W["up"]], 0)
    Yqkv = torch.empty((n, Wqkv.shape[0]), dtype=torch.float32, device=dev)
    Ygu = torch.empty((n, Wgu.shape[0]), dtype=torch.float32, device=dev)

    def step_fused():
        bm.bm_to_f16(x, h, stream=stream)
        bm.bm_f16_matmul(Wqkv, h, Y=Yqkv, stream=stream)
        bm.bm_f16_matmul(W["o"], h, Y=Y["o"], stream=stream)
        bm.bm_f16_matmul(Wgu, h, Y=Ygu, stream=stream)
        bm.bm_to_f16(Y["gate"], hd, stream=stream)  # stand-in FFN activation, same shape as in step()
        bm.bm_f16_matmul(W["down"], hd, Y=Y["down"], stream=stream)

    def step_multi():
        # the same with the separate matrices: bm_f16_matmul_multi shares one launch
        bm.bm_to_f16(x, h, stream=stream)
        bm.bm_f16_matmul_multi([W["q"], W["k"], W["v"]], h, [Y["q"], Y["k"], Y["v"]], stream=stream)
        bm.bm_f16_matmul(W["o"], h, Y=Y["o"], stream=stream)
        bm.bm_f16_matmul_multi([W["gate"], W["up"]], h, [Y["gate"], Y["up"]], stream=stream)
        bm.bm_to_f16(Y["gate"], hd, stream=stream)
        bm.bm_f16_matmul(W["down"], hd, Y=Y["down"], stream=stream)

    old = bm.bm_set_pdl(False)
    try:
        ms_plain = graph_time(torch, stream, step, reps=reps)
        bm.bm_set_pdl(True)
        ms_pdl = graph_time(torch, stream, step, reps=reps)
        ms_fused = graph_time(torch, stream, step_fused, reps=reps)
        ms_multi = graph_time(torch, stream, step_multi, reps=reps)
    finally:
        bm.bm_set_pdl(old)
    res = {"tokens": n, "ms_per_step": round(ms_pdl, 4), "TFLOP_s": round(flops / ms_pdl / 1e9, 1),
           "ms_per_step_without_pdl": round(ms_plain, 4), "TFLOP_s_without_pdl": round(flops / ms_plain / 1e9, 1),
           "how": "one layer's 7 products at 512 columns plus 2 rounding kernels, CUDA graph, PDL on / off",
           "concatenated_weights": {"ms_per_step": round(ms_fused, 4), "TFLOP_s": round(flops / ms_fused / 1e9, 1),
                                    "how": "Q/K/V and gate/up each stored as one matrix: 4 products, PDL on"},
           "multi": {"ms_per_step": round(ms_multi, 4), "TFLOP_s": round(flops / ms_multi / 1e9, 1),
                     "how": "separate matrices, Q/K/V and gate/up through bm_f16_matmul_multi, PDL on"}}
    del W, Y, Wqkv, Wgu, Yqkv, Ygu
    return res


# ----------------------------------------------------------------------------- CPU oracle


def oracle_step_runner():
    """The decode step on the CPU oracle: returns (run_one_step, bytes_per_step)."""
    import oracle

    plan = step_plan()
    tot_bytes = step_bytes(plan, True)  # the same byte count the GPU arm's value uses
    weights = {}
    for op in plan:
        if op[0] != "round":
            for name, rows in op[1]:
                weights[name] = synth.normal_f16(SEED, "smollm2." + name, W_SIGMA, (rows, op[2]))
    acts = {a: synth.normal_f32(SEED, "smollm2.act%d" % a, A_SIGMA, n) for a, n in act_sizes(plan).items()}

    def run():
        h = {}
        for op in plan:
            if op[0] == "round":
                h[op[2]] = oracle.to_f16(acts[op[2]])
            elif op[0] == "multi":
                oracle.matvec_multi([weights[n] for n, _ in op[1]], h[op[3]])
            elif op[0] == "mv":
                oracle.matvec(weights[op[1][0][0]], h[op[3]])
            else:
                oracle.matmul(weights[op[1][0][0]], h[op[3]][None, :])

    return run, tot_bytes, oracle.threads()


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
    run, nbytes, cores = oracle_step_runner()

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
            "sample": "%d full SmolLM2-135M decode steps (30 layers + logits, 269 MB of f16 weights each) "
                      "in %.1f s on the host" % (n, dt),
            "value_1core": round(nbytes * n1 / dt1 / 1e9, 4),
            "sample_1core": "%d full steps in %.1f s on one core" % (n1, dt1), "host": host_cpu(),
            "products": products}


def step_config(world, no_pdl):
    """The workload description both arms print (the reference arm runs it on the host)."""
    return {"workload": "smollm2_135m_decode_step", "layers": LAYERS, "hidden": HIDDEN, "ffn": FFN,
            "q_rows": Q_ROWS, "kv_rows": KV_ROWS, "vocab": VOCAB, "ncols": 1, "seed": SEED,
            "weight_bytes": int(sum(2 * rows * op[2] for op in step_plan() if op[0] != "round"
                                    for _, rows in op[1])),
            "l2": "inputs larger than L2 (269 MB of weights per step, cyclic)",
            "parallelism": "replicas" if world > 1 else "single GPU", "graph": "CUDA graph of the step",
            "pdl": not no_pdl}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    run, nbytes, cores = oracle_step_runner()
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    value = nbytes / (ms / 1e3) / 1e9
    line = {
        "impl": "reference", "metric": "decode F16 GEMV HBM GB/s (SmolLM2-135M decode step)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 weights, f32 accumulate", "data": "synthetic",
        "config": step_config(1, False),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "%d full decode steps after %d warm-up" % (args.steps, args.warmup)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- main


def run_single(spec: str, reps: int):
    """One product ROWSxKxNCOLS, `reps` times (for profilers; prints nothing timed)."""
    import torch

    import __graft_entry__
    import f16_weight_gemv_gb300 as bm

    __graft_entry__.build()
    rows, k, ncols = (int(v) for v in spec.lower().split("x"))
    dev = torch.device("cuda", 0)
    W = torch.from_numpy(synth.normal_f16(SEED, "single.w", W_SIGMA, (rows, k)).view(np.float16)).to(dev)
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
        call = lambda: bm.bm_rms_norm_mul(x, g, 1e-5, y, h)
    elif name == "get_rows":
        E = (torch.randn(128256, 4096, device=dev, generator=gen) * 0.01).to(torch.float16)
        ids = torch.randint(0, 128256, (512,), device=dev, dtype=torch.int32, generator=gen)
        out = torch.empty(512, 4096, dtype=torch.float32, device=dev)
        call = lambda: bm.bm_f16_get_rows(E, ids, out)
    else:
        raise SystemExit("unknown helper " + name)
    for _ in range(reps):
        call()
    torch.cuda.synchronize()
    print(json.dumps({"helper": name, "reps": reps, "status": bm.bm_device_status()}))
    return 0


def run_prefill(reps: int):
    """The Llama-3-8B-shaped prefill layer (bench_llama_prefill), eagerly, `reps` times with
    programmatic dependent launch on (for profilers; prints nothing timed)."""
    import torch

    import __graft_entry__
    import f16_weight_gemv_gb300 as bm

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    hid, ffn, kv, n = 4096, 14336, 1024, 512
    shapes = [("q", hid, hid), ("k", kv, hid), ("v", kv, hid), ("o", hid, hid), ("gate", ffn, hid),
              ("up", ffn, hid), ("down", hid, ffn)]
    W = {nm: torch.from_numpy(synth.normal_f16(SEED, "llama3_8b." + nm, 0.01, (r, c)).view(np.float16)).to(dev)
         for nm, r, c in shapes}
    x = torch.from_numpy(synth.normal_f32(SEED, "llama3_8b.prefill_x", 1.0, (n, hid))).to(dev)
    h = torch.empty((n, hid), dtype=torch.float16, device=dev)
    Y = {nm: torch.empty((n, r), dtype=torch.float32, device=dev) for nm, r, _ in shapes}
    hd = torch.empty((n, ffn), dtype=torch.float16, device=dev)
    bm.bm_set_pdl(True)
    for _ in range(reps):
        bm.bm_to_f16(x, h)
        for nm in ("q", "k", "v", "o", "gate", "up"):
            bm.bm_f16_matmul(W[nm], h, Y=Y[nm])
        bm.bm_to_f16(Y["gate"], hd)
        bm.bm_f16_matmul(W["down"], hd, Y=Y["down"])
    torch.cuda.synchronize()
    print(json.dumps({"prefill": "llama3_8b layer, 512 tokens", "reps": reps, "status": bm.bm_device_status()}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--single", default=None, help="profile mode: run one product ROWSxKxNCOLS --reps times")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--prefill", action="store_true", help="profile mode: run the Llama-3-8B prefill layer --reps times")
    ap.add_argument("--helper", default=None, choices=["mad", "scale", "norm", "get_rows"],
                    help="profile mode: run one of the helpers --reps times")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-products", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.single:
        return run_single(args.single, args.reps)
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

    gpu_name = torch.cuda.get_device_name()
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    value = r["tot_bytes"] * world / (r["ms"] / 1e3) / 1e9
    achieved = r["tot_bytes"] / (r["ms"] / 1e3) / 1e9
    line = {
        "metric": "decode F16 GEMV HBM GB/s (SmolLM2-135M decode step)",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(r["ms"], 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 weights and activations, f32 accumulate (vec_dot bits)", "data": "synthetic",
        "config": step_config(world, args.no_pdl),
        "pct_of_hbm_peak": round(100.0 * value / world / hbm_peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": ncu_traffic(),
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                     "algorithmic_bytes_per_launch": int(r["tot_bytes"] / r["launches_per_step"]),
                     "kernel": "k_gemv_stream (rounding + one-column GEMV)", "peak_source": peak_src,
                     "launches_per_step": r["launches_per_step"],
                     "how": "the step's only kernel: algorithmic bytes of its launches / CUDA-event time of the "
                            "step graph on the launch stream"},
        "unfused": {"ms_per_step": round(r["ms_unfused"], 5),
                    "value": round(r["unfused_bytes"] / (r["ms_unfused"] / 1e3) / 1e9, 2),
                    "launches_per_step": 2 * r["launches_per_step"],
                    "how": "bm_to_f16 then bm_f16_matvec[_multi] / bm_f16_logits per product"},
        "norm_front_end": {"ms_per_step": round(r["ms_norm"], 5),
                           "value": round((r["tot_bytes"] + 4 * HIDDEN * (2 * LAYERS + 1)) / (r["ms_norm"] / 1e3) / 1e9,
                                          2),
                           "how": "the step with the RMS norm (rms_norm then mul) ahead of Q/K/V, gate/up and the "
                                  "logits fused into those launches (bm_f16_matvec_norm)"},
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": r["clocks"],
        "e2e": {"value": round(r["tot_bytes"] / (r["ms_e2e"] / 1e3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "how": "the step's calls through the Python binding, recorded once with prepare(), captured "
                       "with Prepared.graph() and launched every step; pinned host activations in, logits out, "
                       "every step",
                "replay_value": round(r["tot_bytes"] / (r["ms_e2e_replay"] / 1e3) / 1e9, 2),
                "replay_how": "the same recorded calls replayed one C call per product (no graph)",
                "eager_value": round(r["tot_bytes"] / (r["ms_e2e_eager"] / 1e3) / 1e9, 2),
                "eager_how": "the same with every call made through the wrappers (argument checks each time)"},
        "device": gpu_name,
    }
    if "llama3_8b_decode_step" in r:
        r["llama3_8b_decode_step"]["pct_hbm"] = round(100.0 * r["llama3_8b_decode_step"]["GB_s"] / hbm_peak, 1)
        line["llama3_8b_decode_step"] = r["llama3_8b_decode_step"]
    if "qwen3_0.6b_decode_step" in r:
        r["qwen3_0.6b_decode_step"]["pct_hbm"] = round(100.0 * r["qwen3_0.6b_decode_step"]["GB_s"] / hbm_peak, 1)
        line["qwen3_0.6b_decode_step"] = r["qwen3_0.6b_decode_step"]
    if "helpers" in r:
        for p in r["helpers"]:
            p["pct_hbm"] = round(100.0 * p["GB_s"] / hbm_peak, 1)
        line["helpers"] = r["helpers"]
    if "qwen3_0.6b_prefill_layer" in r:
        pq = r["qwen3_0.6b_prefill_layer"]
        pq["pct_bf16_dense_peak"] = round(100.0 * pq["TFLOP_s"] / float(peaks.get("bf16_tflops", 1900.0)), 1)
        line["qwen3_0.6b_prefill_layer"] = pq
    if "llama3_8b_prefill_layer" in r:
        pf = r["llama3_8b_prefill_layer"]
        pk = float(peaks.get("bf16_tflops", 1900.0))
        pf["pct_bf16_dense_peak"] = round(100.0 * pf["TFLOP_s"] / pk, 1)
        for key in ("multi", "concatenated_weights"):
            if key in pf:
                pf[key]["pct_bf16_dense_peak"] = round(100.0 * pf[key]["TFLOP_s"] / pk, 1)
        line["llama3_8b_prefill_layer"] = pf
    if "products" in r:
        line["products"] = r["products"]
        for p in r["products"]:
            if p["ncols"] <= 64:
                p["pct_hbm"] = round(100.0 * p["GB_s"] / hbm_peak, 1)
            else:
                p["pct_bf16_dense_peak"] = round(100.0 * p["TFLOP_s"] / float(peaks.get("bf16_tflops", 1900.0)), 1)
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
