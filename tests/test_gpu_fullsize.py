"""Parity at the benchmark's full sizes, in the launch configurations bench.py times.

- The decode steps exactly as bench.py runs them (Llama-3-8B-shaped, the headline:
  129 calls over 15 GB of weights; SmolLM2-135M- and Qwen3-0.6B-shaped): every
  bm_f16_matvec_act call captured in one CUDA graph with programmatic dependent
  launch, replayed; every output of the step bit for bit against the oracle
  (page f16.md, Design notes, "vec_dot"; forward.md, Advantages, "Shared activations").
- Llama-3-8B and Qwen3-0.6B one-column products at full size, every row bit for bit.
- Llama-3-8B products at 2-64 columns (decode batches) at full size, every element:
  the exact kernel's bits, the tensor cores within the bound.
- The 512-column tensor-core products at full size, EVERY element within
  4e-6 * sum|w*a| of tinyBLAS's element (f16.md, Design notes, "sgemm_dot"), into
  NaN-filled outputs, in the plan the library chooses and again with balanced k
  ranges forced; and the Llama-3-8B prefill layer exactly as bench.py graphs it
  (PDL, split-k reductions, bm_f16_matmul_multi, the other variants beside it).
The oracle's results of a shape are computed once (all host cores) and reused.
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

TOL = 4e-6


def run_step_as_benchmarked(bm, model):
    """bench.py's decode step: built the same way, captured as one graph with PDL on,
    replayed three times into NaN-filled outputs."""
    import torch
    import bench

    s = torch.cuda.Stream()
    old = bm.bm_set_pdl(True)
    try:
        step = bench.DecodeStep(bm, torch, torch.device("cuda"), model, keep_host=True)
        g = bench.capture(torch, s, lambda: step.run(s))
        for o in step.outs.values():
            o.fill_(float("nan"))
        for _ in range(3):
            with torch.cuda.stream(s):
                g.replay()
        torch.cuda.synchronize()
    finally:
        bm.bm_set_pdl(old)
    return step


@pytest.mark.parametrize("model", ["llama3_8b", "smollm2_135m", "qwen3_0.6b"])
def test_decode_step_as_benchmarked(bm, model):
    step = run_step_as_benchmarked(bm, model)
    checked = 0
    for kind, mats, k, a in step.plan:
        off, _ = step.offs[a]
        h = oracle.to_f16(step.act_host[off:off + k])
        for key, wn, _ in mats:
            want = oracle.matvec(step.host_w[wn], h)
            assert np.array_equal(bits32(step.outs[key]), bits32(want)), (model, key)
            checked += want.size
    assert checked == sum(r for _, m, _, _ in step.plan for _, _, r in m)
    assert bm.bm_device_status() == 0
    del step
    import torch
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,rows,k,sigma", [
    ("llama3_8b.q", 4096, 4096, 0.01), ("llama3_8b.down", 4096, 14336, 0.01),
    ("llama3_8b.output", 128256, 4096, 0.01), ("qwen3_0.6b.logits", 151936, 1024, 0.02),
])
def test_full_size_one_column_every_row(bm, name, rows, k, sigma):
    W = synth.normal_f16(0, name, sigma, (rows, k))
    xf = synth.normal_f32(0, name + ".x", 1.0, k)
    y = bm.bm_f16_matvec_act([to_dev(W)], to_dev(xf))[0]
    assert np.array_equal(bits32(y), bits32(oracle.matvec(W, oracle.to_f16(xf))))


# ----------------------------------------------------------------------------- 512 columns, every element


class Reference:
    """W, X and the oracle's Y and sum|w*a| for one product, computed once."""

    def __init__(self, W, X):
        self.W, self.X = W, X
        self.ref = oracle.matmul(W, X).astype(np.float64)
        self.bound = TOL * oracle.abs_matmul(W, X)

    def check(self, Y, what):
        got = Y.detach().cpu().numpy().astype(np.float64) if hasattr(Y, "detach") else Y
        assert np.isfinite(got).all(), what + ": an element was never written (NaN left)"
        err = np.abs(got - self.ref)
        bad = err > self.bound
        assert not bad.any(), "%s: %d elements outside the bound, worst ratio %.3g" % (
            what, int(bad.sum()), float((err / np.maximum(self.bound, 1e-300)).max()))

    def check_cols(self, Y, nc, what):
        """The first nc columns (a product over X[:nc]) within the bound."""
        got = Y.detach().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), what + ": an element was never written (NaN left)"
        err = np.abs(got - self.ref[:nc])
        bad = err > self.bound[:nc]
        assert not bad.any(), "%s: %d elements outside the bound" % (what, int(bad.sum()))

    def bits_cols(self, nc):
        """tinyBLAS's bits of the first nc columns (the oracle's f32 result)."""
        return self.ref[:nc].astype(np.float32).view(np.uint32)


_prefill_refs = {}


def prefill_reference(name):
    """The prefill layer's products (shared by the single-product and the layer tests)."""
    if name not in _prefill_refs:
        _prefill_refs[name] = Reference(*prefill_inputs(name))
    return _prefill_refs[name]


def prefill_inputs(name):
    """The product's W and activation as bench.py's prefill layer draws them."""
    import bench
    shapes = {nm: (r, c) for nm, r, c in bench.PrefillLayer.SHAPES}
    r, c = shapes[name]
    W = synth.normal_f16(0, "llama3_8b." + name, 0.01, (r, c))
    xname = "llama3_8b.prefill_ffn" if name == "down" else "llama3_8b.prefill_x"
    X = oracle.to_f16(synth.normal_f32(0, xname, 1.0, (512, c)))
    return W, X


def other_inputs(name, rows, k):
    W = synth.normal_f16(0, name, 0.02, (rows, k))
    X = oracle.to_f16(synth.normal_f32(0, name + ".X", 1.0, (512, k)))
    return W, X


FULL = [("llama3_8b.q", 4096, 4096), ("llama3_8b.gate", 14336, 4096), ("llama3_8b.down", 4096, 14336),
        ("llama3_8b.output", 128256, 4096), ("qwen3_0.6b.logits", 151936, 1024)]


@pytest.mark.parametrize("name,rows,k", FULL)
def test_full_size_512_columns_every_element(bm, name, rows, k):
    """Every element of the full-size product, in the default plan and with balanced k
    ranges forced, into NaN-filled outputs (a tile never written, or a piece of a
    balanced range dropped, shows as NaN or as an error far outside the bound)."""
    import torch
    short = name.split(".", 1)[1]
    if name.startswith("llama3_8b.") and short in ("q", "gate", "down"):
        ref = prefill_reference(short)
    else:
        ref = Reference(*other_inputs(name, rows, k))
    dW, dX = to_dev(ref.W), to_dev(ref.X)
    plans = []
    for mode in (-1, 1):
        old = bm.bm_set_stream_k(mode)
        try:
            plans.append(bm.bm_tc_plan(rows, k, 512))
            for _ in range(2):  # twice: a second launch finds the first one's workspace contents
                Y = torch.full((512, rows), float("nan"), dtype=torch.float32, device="cuda")
                bm.bm_f16_matmul(dW, dX, Y)
                ref.check(Y, "%s, stream-K mode %d, plan %s" % (name, mode, plans[-1]))
        finally:
            bm.bm_set_stream_k(old)
    assert bm.bm_device_status() == 0
    assert plans[1]["balanced"] == 1, plans  # the forced mode really ran balanced k ranges


FEW = [("q", 4096, 4096), ("gate", 14336, 4096), ("down", 4096, 14336), ("qkv", 6144, 4096)]


@pytest.mark.parametrize("name,rows,k", FEW)
def test_full_size_few_columns_every_element(bm, name, rows, k):
    """Decode-batch widths of the Llama-3-8B products at full size, every element into
    NaN-filled outputs, twice: 2 and 3 columns on the exact CUDA-core kernel, tinyBLAS's
    bits (f16.md, Design notes, "sgemm_dot"; 3 columns with bm_set_exact_sgemm_cols(8)),
    in the consumer layout its launch picks for these row counts; 8, 16 and 64 columns on
    the tensor cores within the bound, where Q and down split k (partials summed in split
    order by the reduction kernel)."""
    import torch
    if name == "qkv":
        W, X = other_inputs("llama3_8b.qkv", rows, k)
        ref = Reference(W, X[:64])
    else:
        ref = prefill_reference(name)
    dW, dX = to_dev(ref.W), to_dev(ref.X)
    plans = {}
    for nc, exact in ((2, 2), (3, 8), (8, 2), (16, 2), (64, 2)):
        old = bm.bm_set_exact_sgemm_cols(exact)
        try:
            Xn = dX[:nc].contiguous()
            if nc > exact:
                plans[nc] = bm.bm_tc_plan(rows, k, nc)
            for _ in range(2):  # twice: the second launch finds the first one's workspace contents
                Y = torch.full((nc, rows), float("nan"), dtype=torch.float32, device="cuda")
                bm.bm_f16_matmul(dW, Xn, Y)
                if nc <= exact:
                    assert np.array_equal(bits32(Y), ref.bits_cols(nc)), (name, nc)
                else:
                    ref.check_cols(Y, nc, "%s x %d columns, plan %s" % (name, nc, plans[nc]))
        finally:
            bm.bm_set_exact_sgemm_cols(old)
    assert bm.bm_device_status() == 0
    if name in ("q", "down"):
        assert all(p["splits"] > 1 for p in plans.values()), plans  # the split-k path ran


@pytest.mark.parametrize("variant", ["multi", "separate", "concat"])
def test_prefill_layer_as_benchmarked(bm, variant):
    """bench.py's Llama-3-8B prefill layer (512 tokens), captured as one CUDA graph with
    PDL on and replayed twice into NaN-filled outputs; every element of all 7 products
    within the bound.  The 'multi' variant is the bench line's prefill value."""
    import torch
    import bench

    s = torch.cuda.Stream()
    old = bm.bm_set_pdl(True)
    try:
        layer = bench.PrefillLayer(bm, torch, torch.device("cuda"))
        g = bench.capture(torch, s, lambda: layer.run(s, variant))
        for Y in layer.Y.values():
            Y.fill_(float("nan"))
        if layer._cat is not None:
            layer._cat[2].fill_(float("nan"))
            layer._cat[3].fill_(float("nan"))
        for _ in range(2):
            with torch.cuda.stream(s):
                g.replay()
        torch.cuda.synchronize()
    finally:
        bm.bm_set_pdl(old)
    # the rounded activations are the oracle's (bit for bit), so the oracle's inputs are its own
    assert np.array_equal(layer.h.cpu().numpy().view(np.uint16), prefill_inputs("q")[1])
    assert np.array_equal(layer.hd.cpu().numpy().view(np.uint16), prefill_inputs("down")[1])
    outs = dict(layer.Y)
    if variant == "concat":
        Yqkv, Ygu = layer._cat[2], layer._cat[3]
        outs.update(q=Yqkv[:, :4096], k=Yqkv[:, 4096:5120], v=Yqkv[:, 5120:], gate=Ygu[:, :14336],
                    up=Ygu[:, 14336:])
    for nm, r, c in bench.PrefillLayer.SHAPES:
        ref = prefill_reference(nm)
        ref.check(outs[nm].contiguous(), "prefill %s, %s" % (variant, nm))
    assert bm.bm_device_status() == 0
    del layer
    torch.cuda.empty_cache()
