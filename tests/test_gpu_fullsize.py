"""Parity at the benchmark's full sizes, in the launch configuration bench.py times.

- The SmolLM2-135M-shaped decode step exactly as bench.py runs it: 121 fused
  bm_f16_matvec_act calls captured in a CUDA graph with programmatic dependent
  launch, replayed; every one of the step's outputs bit for bit against the oracle.
- Llama-3-8B and Qwen3-0.6B one-column products at full size, every row bit for bit.
- Their 512-column tensor-core products on sampled elements, within the bound.
"""
import os
import sys

import numpy as np
import pytest

import oracle
import synth
from conftest import ROOT, bits32, to_dev

pytestmark = pytest.mark.gpu

if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_smollm2_decode_step_as_benchmarked(bm):
    import torch
    import bench

    plan = bench.step_plan()
    dev = torch.device("cuda")
    weights, host_w = {}, {}
    for op in plan:
        if op[0] != "round":
            for name, rows in op[1]:
                w = synth.normal_f16(bench.SEED, "smollm2." + name, bench.W_SIGMA, (rows, op[2]))
                host_w[name] = w
                weights[name] = to_dev(w)
    sizes = bench.act_sizes(plan)
    acts = {a: synth.normal_f32(bench.SEED, "smollm2.act%d" % a, bench.A_SIGMA, n) for a, n in sizes.items()}
    dacts = {a: to_dev(v) for a, v in acts.items()}
    outs = {n: torch.full((w.shape[0],), float("nan"), dtype=torch.float32, device=dev) for n, w in weights.items()}
    s = torch.cuda.Stream()

    def step():
        for op in plan:
            if op[0] == "round":
                continue
            kind, mats, k, a = op
            bm.bm_f16_matvec_act([weights[n] for n, _ in mats], dacts[a], [outs[n] for n, _ in mats], stream=s)

    old = bm.bm_set_pdl(True)
    try:
        with torch.cuda.stream(s):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        for o in outs.values():
            o.fill_(float("nan"))
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
    finally:
        bm.bm_set_pdl(old)
    for op in plan:
        if op[0] == "round":
            continue
        h = oracle.to_f16(acts[op[3]])
        for name, _ in op[1]:
            assert np.array_equal(bits32(outs[name]), bits32(oracle.matvec(host_w[name], h))), name
    assert bm.bm_device_status() == 0


@pytest.mark.parametrize("name,rows,k,sigma", [
    ("llama3_8b.q", 4096, 4096, 0.01), ("llama3_8b.down", 4096, 14336, 0.01),
    ("llama3_8b.output", 128256, 4096, 0.01), ("qwen3_0.6b.logits", 151936, 1024, 0.02),
])
def test_full_size_one_column_every_row(bm, name, rows, k, sigma):
    W = synth.normal_f16(0, name, sigma, (rows, k))
    xf = synth.normal_f32(0, name + ".x", 1.0, k)
    y = bm.bm_f16_matvec_act([to_dev(W)], to_dev(xf))[0]
    assert np.array_equal(bits32(y), bits32(oracle.matvec(W, oracle.to_f16(xf))))


@pytest.mark.parametrize("name,rows,k", [("llama3_8b.gate", 14336, 4096), ("llama3_8b.output", 128256, 4096),
                                         ("qwen3_0.6b.logits", 151936, 1024)])
def test_full_size_512_columns_sampled(bm, name, rows, k):
    W = synth.normal_f16(0, name, 0.01, (rows, k))
    X = oracle.to_f16(synth.normal_f32(0, name + ".X", 1.0, (512, k)))
    Y = bm.bm_f16_matmul(to_dev(W), to_dev(X)).cpu().numpy()
    rng = np.random.default_rng(rows)
    ri = np.concatenate([[0, rows - 1, rows // 2], rng.integers(0, rows, 3000)])
    ci = np.concatenate([[0, 511, 255], rng.integers(0, 512, 3000)])
    ref, ab = oracle.matmul_sample(W, X, ri, ci)
    err = np.abs(Y[ci, ri].astype(np.float64) - ref.astype(np.float64))
    assert (err <= 4e-6 * ab).all(), float((err / ab).max())
