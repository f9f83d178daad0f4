"""Recorded decode steps (bm_step_create / bm_step_run): one launch runs a step's
one-column products in order, each bm_f16_matvec_act's bits (page f16.md, Design
notes, "Activation" and "vec_dot").

- The three decode steps bench.py measures (Llama-3-8B-, Qwen3-0.6B- and
  SmolLM2-135M-shaped), recorded and run twice into NaN-filled outputs: every
  output bit for bit against the oracle.
- A chain in which every call's activation is the previous call's output (and one
  call reads an output two calls back): the kernel's wait between calls must hold,
  or a call would read a stale activation; checked bit for bit against the oracle
  run call after call, over three runs (the step's counter returns to zero).
- The step inside a captured CUDA graph.
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


@pytest.mark.parametrize("model", ["llama3_8b", "qwen3_0.6b", "smollm2_135m"])
def test_recorded_decode_step(bm, model):
    import torch
    import bench

    st = bench.DecodeStep(bm, torch, torch.device("cuda"), model, keep_host=True)
    step = st.record()
    s = torch.cuda.Stream()
    want = {}
    for kind, mats, k, a in st.plan:
        off, _ = st.offs[a]
        h = oracle.to_f16(st.act_host[off:off + k])
        for key, wn, _ in mats:
            want[key] = bits32(oracle.matvec(st.host_w[wn], h))
    for _ in range(2):
        for o in st.outs.values():
            o.fill_(float("nan"))
        step.run(s)
        s.synchronize()
        for key, w in want.items():
            assert np.array_equal(bits32(st.outs[key]), w), (model, key)
    assert bm.bm_device_status() == 0
    step.close()
    del st
    torch.cuda.empty_cache()


def test_each_call_reads_the_outputs_before_it(bm):
    import torch
    dev = torch.device("cuda")
    ks = [1024, 2048, 1024, 512, 4096, 1024, 1024, 2048] * 5
    # call i multiplies W_i (n_{i+1} x k_i; call i+1's k rows) by x_i, where x_0 is an input and
    # x_i (i >= 1) is call i-1's first output; call i's second matrix writes a side output
    Ws, Vs, xs, ys, zs, host = [], [], [], [], [], []
    x0 = synth.normal_f32(0, "step.chain.x0", 1.0, ks[0])
    xs.append(torch.from_numpy(x0).to(dev))
    for i, k in enumerate(ks):
        n = ks[i + 1] if i + 1 < len(ks) else 1000
        W = synth.normal_f16(0, "step.chain.w%d" % i, 1.0 / np.sqrt(k), (n, k))
        V = synth.normal_f16(0, "step.chain.v%d" % i, 0.02, (24, k))
        host.append((W, V))
        Ws.append(to_dev(W))
        Vs.append(to_dev(V))
        ys.append(torch.full((n,), float("nan"), dtype=torch.float32, device=dev))
        zs.append(torch.full((24,), float("nan"), dtype=torch.float32, device=dev))
        if i + 1 < len(ks):
            xs.append(ys[-1])  # the next call's activation is this call's output
    calls = [([Ws[i], Vs[i]], xs[i], [ys[i], zs[i]]) for i in range(len(ks))]
    # one more call reads an output two calls back
    Wb = synth.normal_f16(0, "step.chain.back", 0.02, (40, ks[-2]))
    yb = torch.full((40,), float("nan"), dtype=torch.float32, device=dev)
    calls.append(([to_dev(Wb)], ys[-3], [yb]))
    step = bm.bm_step_create(calls)

    # the oracle, call after call
    x = x0
    want_y, want_z = [], []
    for i, (W, V) in enumerate(host):
        h = oracle.to_f16(x)
        want_y.append(oracle.matvec(W, h))
        want_z.append(oracle.matvec(V, h))
        x = want_y[-1]
    want_b = oracle.matvec(Wb, oracle.to_f16(want_y[-3]))
    assert all(np.isfinite(w).all() for w in want_y)

    s = torch.cuda.Stream()
    for run in range(3):
        for t in ys + zs + [yb]:
            t.fill_(float("nan"))
        step.run(s)
        s.synchronize()
        for i in range(len(ks)):
            assert np.array_equal(bits32(ys[i]), bits32(want_y[i])), (run, i)
            assert np.array_equal(bits32(zs[i]), bits32(want_z[i])), (run, i)
        assert np.array_equal(bits32(yb), bits32(want_b)), run
    assert bm.bm_device_status() == 0
    step.close()


def test_recorded_step_in_a_cuda_graph(bm):
    import torch
    dev = torch.device("cuda")
    k, n = 2048, 3000
    W1 = synth.normal_f16(0, "step.graph.w1", 1.0 / np.sqrt(k), (k, k))
    W2 = synth.normal_f16(0, "step.graph.w2", 0.02, (n, k))
    x = synth.normal_f32(0, "step.graph.x", 1.0, k)
    dx = torch.from_numpy(x).to(dev)
    y1 = torch.empty(k, dtype=torch.float32, device=dev)
    y2 = torch.empty(n, dtype=torch.float32, device=dev)
    step = bm.bm_step_create([([to_dev(W1)], dx, [y1]), ([to_dev(W2)], y1, [y2])])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.run(s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.run(s)
    want1 = oracle.matvec(W1, oracle.to_f16(x))
    want2 = oracle.matvec(W2, oracle.to_f16(want1))
    for _ in range(2):
        y1.fill_(float("nan"))
        y2.fill_(float("nan"))
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert np.array_equal(bits32(y1), bits32(want1))
        assert np.array_equal(bits32(y2), bits32(want2))
    assert bm.bm_device_status() == 0
    step.close()
